"""Pins of the oracle's accept-rate target (P1 section 3.9 "Accept rate 3D";
P2 section 3.5) and of eval_mask / tau (P1 sections 3.6 and 3.10)."""
import numpy as np
import pytest
from scipy import special

import oracle as O


def test_identical_rows_give_one():
    x = np.random.default_rng(0).normal(0, 3, 1000).astype(np.float32)
    acc, chk = O.tv_row(x, x.copy())
    assert abs(acc - 1.0) < 1e-12 and abs(chk - 1.0) < 1e-12


def test_disjoint_one_hots_give_zero():
    d = np.full(16, -200.0, np.float32)
    t = np.full(16, -200.0, np.float32)
    d[3], t[11] = 200.0, 200.0
    acc, chk = O.tv_row(d, t)
    assert acc < 1e-100 and abs(chk) < 1e-12


def test_sum_min_equals_one_minus_tv_and_softmax():
    rng = np.random.default_rng(1)
    for _ in range(20):
        d = rng.normal(0, 3, 257).astype(np.float32)
        t = (0.8 * d + rng.normal(0, 2, 257)).astype(np.float32)
        acc, chk = O.tv_row(d, t)
        p, q = special.softmax(t.astype(np.float64)), special.softmax(d.astype(np.float64))
        assert abs(acc - chk) < 1e-12
        assert abs(acc - np.minimum(p, q).sum()) < 1e-12


def test_two_point_closed_form():
    for a, b in [(0.3, -1.2), (2.0, 2.0), (-4.0, 5.0)]:
        d = np.array([a, 0.0], np.float32)
        t = np.array([b, 0.0], np.float32)
        acc, _ = O.tv_row(d, t)
        sa, sb = 1 / (1 + np.exp(-np.float64(np.float32(a)))), 1 / (1 + np.exp(-np.float64(np.float32(b))))
        assert abs(acc - (1 - abs(sa - sb))) < 1e-12


def test_permutation_invariance_and_bf16_input():
    rng = np.random.default_rng(2)
    d = rng.normal(0, 3, 300).astype(np.float32)
    t = rng.normal(0, 3, 300).astype(np.float32)
    perm = rng.permutation(300)
    a1, _ = O.tv_row(d, t)
    a2, _ = O.tv_row(d[perm].copy(), t[perm].copy())
    assert abs(a1 - a2) < 1e-12
    db = (d.view(np.uint32) >> 16).astype(np.uint16)  # truncated bf16 patterns
    tb = (t.view(np.uint32) >> 16).astype(np.uint16)
    a3, _ = O.tv_row(db, tb)
    p = special.softmax(O.to_f64(tb))
    q = special.softmax(O.to_f64(db))
    assert abs(a3 - np.minimum(p, q).sum()) < 1e-12


def test_eval_mask_cumprod_and_tau():
    acc = np.array([0.9, 0.5, 0.8, 0.7])
    m, tau = O.eval_mask_tau(acc, 1, None)
    assert np.array_equal(m, np.ones(4))
    assert abs(tau - (1 + 0.9 + 0.45 + 0.36 + 0.252)) < 1e-12
    m, tau = O.eval_mask_tau(acc, 1, np.array([1, 0, 1, 1], np.uint8))
    assert np.array_equal(m, [1, 0, 0, 0]) and abs(tau - 1.9) < 1e-12  # zero after the first zero
    m, tau = O.eval_mask_tau(acc, 0, None)
    assert np.array_equal(m, np.zeros(4)) and tau == 1.0
    m, tau = O.eval_mask_tau(np.ones(8), 1, None)
    assert tau == 9.0


def test_l1_term_is_the_sum_of_absolute_differences():
    # the oracle's route (2 (1 - sum min(p, q)) from the TV row) against the page's definition
    # sum_v |softmax(d) - softmax(t)| written out directly
    rng = np.random.default_rng(11)
    for V in (7, 100, 3000):
        d = rng.normal(0, 2, V).astype(np.float32)
        t = (0.6 * d + rng.normal(0, 1.5, V)).astype(np.float32)
        acc, _ = O.tv_row(d, t)
        p = np.exp(d.astype(np.float64) - d.max())
        p /= p.sum()
        q = np.exp(t.astype(np.float64) - t.max())
        q /= q.sum()
        l1, _, _ = O.tv_l1_loss(np.array([[[acc]]]), np.ones((1, 1, 1)))
        assert abs(l1[0, 0, 0] - np.abs(p - q).sum()) < 1e-12


def test_l1_position_weights():
    gamma, decay = 8, 4.0
    for k in range(gamma):  # one live position: the sums are 2 w_k (accept 0) and w_k
        mask = np.zeros((1, 1, gamma))
        mask[0, 0, k] = 1.0
        _, num, den = O.tv_l1_loss(np.zeros((1, 1, gamma)), mask, decay)
        assert den == pytest.approx(np.exp(-1.0 / decay) ** k, rel=1e-14)
        assert num == pytest.approx(2.0 * den, rel=1e-14)
    _, num, den = O.tv_l1_loss(np.ones((3, 5, gamma)), np.ones((3, 5, gamma)), decay)
    assert num == 0.0 and den == pytest.approx(15 * sum(np.exp(-np.arange(gamma) / decay)))
