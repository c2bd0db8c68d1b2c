"""Pins of the oracle's verify-length selection (P3 section "置信度调度与验证
截断"; survival as a product of conditional confidences, P2 section 3.8.3) and of
the throughput-aware Theta scheduler (P4 section 5.1, worked example)."""
import itertools
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden", "theta_worked_example.txt")


def _survival_f32(conf):
    c = np.clip(np.nan_to_num(conf.astype(np.float32), nan=0.0), 0, 1).astype(np.float32)
    a = np.empty_like(c)
    run = np.ones(c.shape[0], np.float32)
    for i in range(c.shape[1]):
        run = (run * c[:, i]).astype(np.float32)
        a[:, i] = run
    return a


def _brute(conf, budget):
    a = _survival_f32(conf).astype(np.float64)
    B, g = a.shape
    best, arg, nbest = -1.0, None, 0
    for L in itertools.product(range(1, g + 1), repeat=B):
        if sum(L) > budget:
            continue
        v = sum(a[j, :L[j]].sum() for j in range(B))
        if v > best + 1e-15:
            best, arg, nbest = v, L, 1
        elif abs(v - best) <= 1e-15:
            nbest += 1
    return best, arg, nbest


@pytest.mark.parametrize("seed", range(12))
def test_schedule_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    B, g = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    conf = rng.beta(3, 1.5, (B, g)).astype(np.float32)
    for budget in range(B, B * g + 2):
        L, off, obj, mg = O.schedule(conf, budget)
        best, arg, nbest = _brute(conf, budget)
        assert abs(obj - best) < 1e-12
        assert L.sum() <= budget and L.min() >= 1 and L.max() <= g
        assert off[0] == 0 and np.array_equal(np.diff(off), L)
        if nbest == 1:
            assert tuple(L) == arg


def test_schedule_edges():
    rng = np.random.default_rng(3)
    conf = rng.uniform(0, 1, (6, 5)).astype(np.float32)
    L, off, obj, _ = O.schedule(conf, 6)
    assert np.all(L == 1)
    L, off, obj, _ = O.schedule(conf, 30)
    assert np.all(L == 5) and off[-1] == 30
    L, off, obj, _ = O.schedule(conf, 1000)
    assert np.all(L == 5)
    with pytest.raises(ValueError):
        O.schedule(conf, 5)


def test_schedule_ties_are_prefix_closed():
    conf = np.ones((3, 4), np.float32)  # every survival is 1: ties broken by (j asc, i asc)
    L, off, obj, mg = O.schedule(conf, 6)
    assert list(L) == [4, 1, 1] and mg == 0.0
    conf[1, 0] = np.nan  # NaN confidence reads as 0
    L, *_ = O.schedule(conf, 9)
    assert list(L) == [4, 1, 4]


def test_theta_worked_example():
    rows = {}
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        rows[k] = [float(x) for x in v]
    c = np.array(rows["c"] + [0.1])  # c_3 is truncated on the page; any value <= 1 keeps the stop at l = 2
    sps = np.array(rows["sps"])
    ell, th = O.theta_schedule(c, sps)
    assert ell == int(rows["chosen"][0])
    np.testing.assert_allclose(np.round(th[:3], 2), rows["theta"])
    assert np.isnan(th[3])  # the causal search never looked past the first drop
