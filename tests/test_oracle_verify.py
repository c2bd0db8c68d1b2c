"""Pins of the oracle's lossless verification (P3 "Speculative Decoding":
rejection sampling left to right, truncate at the first failure, resample from
the target; the output law equals the target's)."""
import numpy as np
import pytest
from scipy import special, stats

import oracle as O


def _logits(seed, V=8, scale=1.3):
    return np.random.default_rng(seed).normal(0, scale, V).astype(np.float32)


@pytest.mark.parametrize("T", [0.7, 1.0])
def test_accept_probability_is_sum_min(T):
    zd, zt = _logits(1), _logits(2)
    q, p = special.softmax(zd.astype(np.float64) / T), special.softmax(zt.astype(np.float64) / T)
    N = 400_000
    em, na = O.trials_spec_one(zd, zt, T, 3, 21, N, CS=2)
    pa = np.minimum(p, q).sum()
    assert abs(pa - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12
    assert abs(na / N - pa) < 5 * np.sqrt(pa * (1 - pa) / N)


@pytest.mark.parametrize("T,TS,CS", [(1.0, 8, 8), (0.7, 2, 1), (1.0, 3, 2), (1.0, 8, 4)])
def test_emitted_token_law_is_target(T, TS, CS):
    zd, zt = _logits(3), _logits(4)
    p = special.softmax(zt.astype(np.float64) / T)
    em, na = O.trials_spec_one(zd, zt, T, TS, 31 + TS + CS, 1_000_000, CS=CS)
    assert stats.chisquare(em, p * em.sum()).pvalue > 1e-3


def test_emitted_law_rejects_draft_law():
    # the same statistic must reject "emitted ~ q" (a verify that always accepts)
    T = 1.0
    zd, zt = _logits(3), _logits(4)
    q = special.softmax(zd.astype(np.float64) / T)
    em, na = O.trials_spec_one(zd, zt, T, 8, 39, 1_000_000)
    assert stats.chisquare(em, q * em.sum()).pvalue < 1e-6


def test_identical_distributions_always_accept():
    zd = _logits(5)
    N = 200_000
    em, na = O.trials_spec_one(zd, zd.copy(), 1.0, 8, 41, N)
    # q(x) uses the float32-rounded draft LSE: at most a ~1e-7 log-ratio error
    assert na >= N - 2


def test_residual_support_is_where_target_exceeds_draft():
    T = 1.0
    zd, zt = _logits(6), _logits(7)
    q, p = special.softmax(zd.astype(np.float64) / T), special.softmax(zt.astype(np.float64) / T)
    lse_d = np.float32(special.logsumexp(zd.astype(np.float64) / T))
    base = zd.reshape(1, 1, 8)
    tgt = zt.reshape(1, 1, 8)
    seen = set()
    for j in range(3000):
        x, _, _ = O.chunk_gumbel(zd.astype(np.float64) / T, 3, j, 1, CS=4)
        n, corr, mm, fb = O.verify_request(base, None, None, 0, j, np.array([x], np.int32), np.array([lse_d]),
                                           np.array([zd[x]]), tgt, 1, T, 3, 8, row=0, CS=4)
        if n == 0:
            assert p[corr] > q[corr] and fb == 0
            seen.add(corr)
    assert seen == set(np.nonzero(p > q)[0].tolist())


def test_greedy_verify():
    rng = np.random.default_rng(8)
    V, gamma = 16, 3
    base = rng.normal(0, 1, (1, gamma, V)).astype(np.float32)
    tgt = rng.normal(0, 1, (1, gamma + 1, V)).astype(np.float32)
    am = tgt[0].argmax(-1)
    tokens = am[:gamma].astype(np.int32).copy()
    tokens[1] = (tokens[1] + 1) % V  # position 2 disagrees with the target argmax
    n, corr, mm, fb = O.verify_request(base, None, None, 0, 0, tokens, np.zeros(gamma), np.zeros(gamma), tgt,
                                       gamma, 0.0, 0, 1024)
    assert n == 1 and corr == am[1]
    tokens[1] = am[1]
    n, corr, mm, fb = O.verify_request(base, None, None, 0, 0, tokens, np.zeros(gamma), np.zeros(gamma), tgt,
                                       gamma, 0.0, 0, 1024)
    assert n == 3 and corr == am[3]  # all accepted: bonus from target row 4
    n, corr, mm, fb = O.verify_request(base, None, None, 0, 0, tokens, np.zeros(gamma), np.zeros(gamma),
                                       np.ascontiguousarray(tgt[:, :gamma]), gamma, 0.0, 0, 1024)
    assert n == 3 and corr == -1  # no row L+1: no bonus


def _exact_accept_len_law(base, W1, W2, anchor, tgt, T):
    """Independent forward recursion: alpha_1(x) = min(q_1(x|anchor), p_1(x)),
    alpha_k(x) = sum_x' alpha_{k-1}(x') min(q_k(x|x'), p_k(x));
    P(n >= k) = sum_x alpha_k(x)."""
    gamma, V = base.shape
    b, w1, w2, t = (a.astype(np.float64) for a in (base, W1, W2, tgt))
    bias = w1 @ w2.T  # bias[prev, v]
    P = [special.softmax(t[i] / T) for i in range(gamma)]
    q1 = special.softmax((b[0] + bias[anchor]) / T)
    alpha = np.minimum(q1, P[0])
    ge = [1.0, alpha.sum()]
    for i in range(1, gamma):
        Q = special.softmax((b[i][None, :] + bias) / T, axis=1)  # Q[prev, x]
        alpha = (alpha[:, None] * np.minimum(Q, P[i][None, :])).sum(0)
        ge.append(alpha.sum())
    ge.append(0.0)
    return np.array([ge[k] - ge[k + 1] for k in range(gamma + 1)])


@pytest.mark.parametrize("T,TS,CS", [(1.0, 8, 8), (0.7, 3, 2)])
def test_accepted_length_law_exact(T, TS, CS):
    rng = np.random.default_rng(12)
    V, gamma, r = 8, 3, 2
    base = rng.normal(0, 1.0, (gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.9, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.9, (V, r)).astype(np.float32)
    tgt = (base + rng.normal(0, 0.6, (gamma, V))).astype(np.float32)
    law = _exact_accept_len_law(base, W1, W2, 4, tgt, T)
    assert abs(law.sum() - 1) < 1e-12
    hist = O.trials_spec_block(base, W1, W2, 4, tgt, T, TS, 55, 1_000_000, CS=CS)
    assert stats.chisquare(hist, law * hist.sum()).pvalue > 1e-3
    # a plausible mistake (ignoring the Markov bias when verifying) changes the law
    law0 = _exact_accept_len_law(base, W1 * 0, W2, 4, tgt, T)
    assert stats.chisquare(hist, law0 * hist.sum()).pvalue < 1e-6
