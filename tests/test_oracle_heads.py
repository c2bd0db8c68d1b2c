"""Pins of the oracle's Gated and RNN Markov heads (page "03 · DSpark 建模：Markov 与 Confidence",
section 3.7; page "DSpark 深度解读", section 3.3, the table of the three heads):
  gated: gate = sigmoid(Wg [h; W1[x]]),  bias = W2 (gate * W1[x])
  rnn:   z = [s; W1[x]; h],  s <- sigmoid(Wg z) s + (1 - sigmoid(Wg z)) tanh(Wc z),  bias = W2 tanh(Wo z)
Each pin reduces a head to the vanilla head or to a sequence worked out by hand."""
import math

import numpy as np
import pytest

import oracle as O

TS = 64


def setup(B=2, g=4, V=300, r=4, d=3, seed=0):
    rng = np.random.default_rng(seed)
    base = rng.normal(0, 2, (B, g, V)).astype(np.float32)
    W1 = rng.normal(0, 0.8, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.8, (V, r)).astype(np.float32)
    hidden = rng.normal(0, 1, (B, g, d)).astype(np.float32)
    return base, W1, W2, hidden, rng


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_gated_zero_weights_is_vanilla_at_half_gate(T):
    # Wg = 0: gate = sigmoid(0) = 1/2 exactly, so the head is the vanilla head with W1 / 2 (exact in fp32)
    base, W1, W2, hidden, _ = setup()
    r, d = W1.shape[1], hidden.shape[-1]
    Wg = np.zeros((r, d + r), np.float32)
    for j in range(base.shape[0]):
        tok, lse, zx, mg, u = O.sample_request_head(base, W1, W2, 5, j, T, 3, TS, O.HEAD_GATED, hidden, Wg)
        rt, rl, rz, rm = O.sample_request(base, (W1 * 0.5).astype(np.float32), W2, 5, j, T, 3, TS)
        assert np.array_equal(tok, rt) and np.array_equal(zx, rz)
        assert np.array_equal(np.isnan(lse), np.isnan(rl)) and np.allclose(lse, rl, rtol=0, atol=0, equal_nan=True)
        prev = np.concatenate([[5], tok[:-1]])
        assert np.array_equal(u, 0.5 * W1[prev].astype(np.float64))


def test_gated_gate_direction_and_column_order():
    # a pre-activation of ln 3 in the hidden-state columns gives gate = 3/4 (sigmoid(-ln 3) would be 1/4);
    # the W1 columns of Wg stay zero, so only the [h; W1[x]] order puts the weight on h
    base, W1, W2, hidden, _ = setup(B=1)
    r, d = W1.shape[1], hidden.shape[-1]
    hidden = np.zeros_like(hidden)
    hidden[..., 1] = 1.0
    Wg = np.zeros((r, d + r), np.float32)
    Wg[:, 1] = np.float32(math.log(3.0))
    tok, lse, zx, mg, u = O.sample_request_head(base, W1, W2, 9, 0, 1.0, 4, TS, O.HEAD_GATED, hidden, Wg)
    prev = np.concatenate([[9], tok[:-1]])
    assert np.allclose(u, 0.75 * W1[prev].astype(np.float64), rtol=1e-7, atol=0)
    rt, rl, rz, rm = O.sample_request(base, (W1 * 0.75).astype(np.float32), W2, 9, 0, 1.0, 4, TS)
    ok = rm > 1e-5
    assert np.array_equal(tok[ok], rt[ok]) and np.allclose(lse, rl, rtol=1e-7)


def test_gated_saturated_gates():
    base, W1, W2, hidden, _ = setup(B=1)
    r, d = W1.shape[1], hidden.shape[-1]
    hidden = np.ones_like(hidden)
    Wg = np.zeros((r, d + r), np.float32)
    Wg[:, 0] = 1e30  # gate = 1 exactly: the vanilla head
    got = O.sample_request_head(base, W1, W2, 2, 0, 1.0, 1, TS, O.HEAD_GATED, hidden, Wg)
    ref = O.sample_request(base, W1, W2, 2, 0, 1.0, 1, TS)
    for a, b in zip(got[:4], ref):
        assert np.array_equal(np.nan_to_num(a, nan=7.0), np.nan_to_num(b, nan=7.0))
    Wg[:, 0] = -1e30  # gate = 0: no bias, the DFlash draft of the base logits alone
    got = O.sample_request_head(base, W1, W2, 2, 0, 1.0, 1, TS, O.HEAD_GATED, hidden, Wg)
    ref = O.sample_request(base, None, None, 2, 0, 1.0, 1, TS)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[2], ref[2]) and not got[4].any()


def test_rnn_state_sequence_by_hand():
    # r = 2, d = 1, h = 1: Wg = 0 (gate 1/2), Wc reads h with weight atanh(1/2) (candidate 1/2), Wo reads the
    # state itself.  From s_0 = 0: s_k = s_{k-1} / 2 + 1/4, i.e. 0, 1/4, 3/8, 7/16, ..., and the bias of step k
    # uses z_k, which holds s_{k-1}: u_k = tanh(s_{k-1}) = tanh((1 - 2^-(k-1)) / 2).
    g, V, r, d = 5, 40, 2, 1
    base, W1, W2, _, _ = setup(B=1, g=g, V=V, r=r, d=d, seed=2)
    hidden = np.ones((1, g, d), np.float32)
    w = 2 * r + d
    Wg = np.zeros((r, w), np.float32)
    Wc = np.zeros((r, w), np.float32)
    Wc[:, 2 * r] = np.float32(math.atanh(0.5))
    Wo = np.zeros((r, w), np.float32)
    Wo[0, 0] = Wo[1, 1] = 1.0
    tok, lse, zx, mg, u = O.sample_request_head(base, W1, W2, 1, 0, 0.0, 0, TS, O.HEAD_RNN, hidden, Wg, Wc, Wo)
    for k in range(1, g + 1):
        want = math.tanh((1.0 - 2.0 ** -(k - 1)) / 2.0)
        assert np.allclose(u[k - 1], want, rtol=0, atol=2e-8), (k, u[k - 1], want)
    # the drafted tokens follow the bias W2 u_k (greedy)
    for k in range(g):
        z = base[0, k].astype(np.float64) + W2.astype(np.float64) @ u[k]
        assert tok[k] == int(np.argmax(z)) and zx[k] == z[tok[k]]


def test_rnn_without_output_weights_is_dflash():
    base, W1, W2, hidden, rng = setup(B=1)
    r, d = W1.shape[1], hidden.shape[-1]
    w = 2 * r + d
    Wg = rng.normal(0, 1, (r, w)).astype(np.float32)
    Wc = rng.normal(0, 1, (r, w)).astype(np.float32)
    Wo = np.zeros((r, w), np.float32)
    got = O.sample_request_head(base, W1, W2, 4, 0, 1.0, 6, TS, O.HEAD_RNN, hidden, Wg, Wc, Wo)
    ref = O.sample_request(base, None, None, 4, 0, 1.0, 6, TS)
    assert np.array_equal(got[0], ref[0]) and np.allclose(got[1], ref[1], rtol=1e-15) and not got[4].any()


def test_verify_with_head_vectors_matches_the_equivalent_vanilla_head():
    # the half-gate head of the first pin, verified with its head vectors, is the vanilla head with W1 / 2
    base, W1, W2, hidden, rng = setup(B=3, g=3, V=200)
    r, d = W1.shape[1], hidden.shape[-1]
    target = (base + rng.normal(0, 1.0, base.shape)).astype(np.float32)
    Wg = np.zeros((r, d + r), np.float32)
    for j in range(3):
        tok, lse, zx, mg, u = O.sample_request_head(base, W1, W2, 7, j, 1.0, 11, TS, O.HEAD_GATED, hidden, Wg)
        got = O.verify_request(base, W1, W2, 7, j, tok, lse.astype(np.float32), zx.astype(np.float32), target, 3, 1.0,
                               11, TS, head_vec=u)
        ref = O.verify_request(base, (W1 * 0.5).astype(np.float32), W2, 7, j, tok, lse.astype(np.float32),
                               zx.astype(np.float32), target, 3, 1.0, 11, TS)
        assert got == ref
