"""Pins of the oracle's verify-length selection (P3 section "置信度调度与验证
截断"; survival as a product of conditional confidences, P2 section 3.8.3) and of
the throughput-aware Theta scheduler (P4 section 5.1, worked example)."""
import itertools
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden", "theta_worked_example.txt")


def _survival(conf):
    # prefix products of the clamped conditional confidences, in double (the definition)
    c = np.clip(np.nan_to_num(conf.astype(np.float64), nan=0.0), 0, 1)
    return np.cumprod(c, axis=1)


def _brute(conf, budget):
    a = _survival(conf)
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


def test_schedule_survival_is_double_precision():
    # two requests whose second-position survivals c1*c2 are equal once rounded to fp32 but differ
    # in double: with one extra verify slot the larger true product must win, not the lower index
    rng = np.random.default_rng(0)
    x = rng.uniform(0.5, 1.0, (200000, 2)).astype(np.float32)
    p32 = (x[:, 0] * x[:, 1]).astype(np.float32)
    p64 = x[:, 0].astype(np.float64) * x[:, 1].astype(np.float64)
    order = np.argsort(p32, kind="stable")
    found = None
    for k in range(len(order) - 1):
        a, b = order[k], order[k + 1]
        if p32[a] == p32[b] and p64[a] != p64[b]:
            lo, hi = (a, b) if p64[a] < p64[b] else (b, a)
            found = (lo, hi)
            break
    assert found is not None
    lo, hi = found
    conf = np.stack([x[lo], x[hi]]).astype(np.float32)  # row 0 has the smaller true product
    L, off, obj, mg = O.schedule(conf, 3)
    assert list(L) == [1, 2]
    assert mg == p64[hi] - p64[lo] and 0 < mg < 1e-7
    assert abs(obj - (float(conf[0, 0]) + float(conf[1, 0]) + p64[hi])) < 1e-15


def test_schedule_margin_is_the_boundary_gap():
    conf = np.array([[1.0, 0.9, 0.5], [1.0, 0.6, 0.5]], np.float32)
    # candidates (a desc): 0.9 (j0,i2), 0.6 (j1,i2), 0.45 (j0,i3), 0.3 (j1,i3); budget 3 takes one
    L, off, obj, mg = O.schedule(conf, 3)
    assert list(L) == [2, 1]
    assert abs(mg - (0.9 - 0.6)) < 1e-7
    L, off, obj, mg = O.schedule(conf, 6)  # everything taken: nothing left to compare
    assert list(L) == [3, 3] and mg == np.inf


def test_theta_margin_and_double_precision():
    # the worked example: the search compares Theta_1 with Theta_0 and Theta_2 with Theta_1
    ell, th, mg = O.theta_schedule(np.array([0.8, 0.7, 0.1]), np.array([1.0, 0.95, 0.52, 0.48]), with_margin=True)
    t0, t1, t2 = 1.0, 1.8 * 0.95, 2.36 * 0.52
    assert ell == 1
    assert abs(mg - min((t1 - t0) / t1, (t1 - t2) / t1)) < 1e-12
    # Theta_1 = 1.25 (0.8 - 1e-12) lies 1.25e-12 below Theta_0 = 1: the search stops at once.  In
    # single precision the two would round to the same value and the search would go on.
    ell, th, mg = O.theta_schedule(np.array([0.25, 0.0]), np.array([1.0, 0.8 - 1e-12, 0.1]), with_margin=True)
    assert ell == 0 and np.isnan(th[2])
    assert abs(mg - 1.25e-12) < 1e-15
    # a search that never stops reports the smallest gap it saw; gamma = 0 compares nothing
    ell, th, mg = O.theta_schedule(np.array([0.5, 0.5]), np.array([1.0, 1.0, 1.0]), with_margin=True)
    assert ell == 2 and abs(mg - 0.25 / 1.75) < 1e-12
    ell, th, mg = O.theta_schedule(np.zeros(0), np.array([2.0]), with_margin=True)
    assert ell == 0 and th[0] == 2.0 and mg == np.inf


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
