"""Pins of the oracle's Markov head and samplers against closed forms, library
routines on tiny inputs, and chi-square on V=8 (P2 section 3.4; P1 section 3.7)."""
import numpy as np
import pytest
from scipy import special, stats

import oracle as O


def _bf16(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = a.view(np.uint32)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def test_markov_r0_is_identity():
    rng = np.random.default_rng(0)
    base = rng.normal(0, 2, 16).astype(np.float32)
    z = O.markov_logits(base, None, None, 3)
    assert np.array_equal(z, base.astype(np.float64))


def test_markov_one_hot_w1_reads_one_w2_column():
    rng = np.random.default_rng(1)
    V, r = 10, 4
    base = rng.normal(0, 1, V).astype(np.float32)
    W1 = np.zeros((V, r), np.float32)
    W1[6, 2] = 1.0
    W2 = rng.normal(0, 1, (V, r)).astype(np.float32)
    z = O.markov_logits(base, W1, W2, 6)
    np.testing.assert_array_equal(z, base.astype(np.float64) + W2[:, 2].astype(np.float64))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_markov_matches_matmul(dt):
    rng = np.random.default_rng(2)
    V, r = 8, 2
    base = rng.normal(0, 3, V).astype(np.float32)
    W1 = rng.normal(0, 0.5, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.5, (V, r)).astype(np.float32)
    if dt == "bf16":
        base, W1, W2 = _bf16(base), _bf16(W1), _bf16(W2)
    for prev in range(V):
        z = O.markov_logits(base, W1, W2, prev)
        ref = O.to_f64(base) + O.to_f64(W2) @ O.to_f64(W1)[prev]
        np.testing.assert_allclose(z, ref, rtol=0, atol=1e-14)


def test_argmax_lowest_index_on_ties():
    z = np.array([1.0, 3.0, 2.0, 3.0])
    x, m = O.argmax(z)
    assert x == 1 and m == 0.0
    z = np.array([0.5, -1.0, 2.0])
    assert O.argmax(z) == (2, 1.5)
    rng = np.random.default_rng(3)
    for _ in range(50):
        z = rng.normal(size=33)
        assert O.argmax(z)[0] == int(np.argmax(z))


def test_single_chunk_is_inverse_cdf():
    rng = np.random.default_rng(4)
    lw = rng.normal(0, 1.5, 8)
    p = special.softmax(lw)
    cdf = np.cumsum(p)
    for j in range(200):
        # a vocabulary of one chunk: the draft draw and the corrections' draw (their own purposes)
        for pc, pin in ((O.P_SAMPLE_CHUNK, O.P_SAMPLE_INCHUNK), (O.P_RESID_CHUNK, O.P_RESID_INCHUNK),
                        (O.P_BONUS_CHUNK, O.P_BONUS_INCHUNK)):
            x, m, lse = O.chunk_gumbel(lw, 5, j, 2, CS=8, p_chunk=pc, p_inchunk=pin)
            u = O.uniform(5, j, 2, pin, 0)
            assert x == int(np.searchsorted(cdf, u, side="right"))
            assert abs(lse - special.logsumexp(lw)) < 1e-12


def test_chunk_race_then_inverse_cdf():
    # 12 ids in chunks of 4: the chunk with the largest LSE_c - ln(-ln u_c) wins, the id is the
    # in-order inverse CDF of u inside it; the short last chunk (V = 14) takes part too
    rng = np.random.default_rng(15)
    for V in (12, 14):
        lw = rng.normal(0, 1.0, V)
        nc = (V + 3) // 4
        lse_c = np.array([special.logsumexp(lw[4 * c:4 * c + 4]) for c in range(nc)])
        for j in range(300):
            x, m, lse = O.chunk_gumbel(lw, 7, j, 3, CS=4)
            keys = [lse_c[c] - np.log(-np.log(O.uniform(7, j, 3, O.P_SAMPLE_CHUNK, c))) for c in range(nc)]
            c = int(np.argmax(keys))
            u = O.uniform(7, j, 3, O.P_SAMPLE_INCHUNK, 0)
            pc = special.softmax(lw[4 * c:4 * c + 4])
            k = int(np.searchsorted(np.cumsum(pc), u, side="right"))
            assert x == 4 * c + k
            assert m <= sorted(keys)[-1] - sorted(keys)[-2] + 1e-12


def test_chunk_sampler_skips_zero_mass():
    lw = np.array([-np.inf, -np.inf, 0.3, 1.0, -np.inf, -np.inf, -np.inf, -2.0, -np.inf])
    for j in range(300):
        x, m, lse = O.chunk_gumbel(lw, 9, j, 1, CS=2)
        assert np.isfinite(lw[x])
    assert abs(lse - special.logsumexp(lw)) < 1e-12
    assert O.chunk_gumbel(np.full(5, -np.inf), 1, 0, 1, CS=2)[0] == -1


def test_corrections_race_with_their_own_purposes():
    # the residual draw races chunks on E_c = -ln U(RESID_CHUNK, c) and draws inside the winner with
    # U(RESID_INCHUNK, 0): the same contract as the draft draw with the other purposes
    rng = np.random.default_rng(14)
    lw = rng.normal(0, 1.0, 12)
    lw[5] = -np.inf
    lse_c = np.array([special.logsumexp(lw[4 * c:4 * c + 4]) for c in range(3)])
    for j in range(300):
        x, m, lse = O.chunk_gumbel(lw, 6, j, 3, CS=4, p_chunk=O.P_RESID_CHUNK, p_inchunk=O.P_RESID_INCHUNK)
        keys = [lse_c[c] - np.log(-np.log(O.uniform(6, j, 3, O.P_RESID_CHUNK, c))) for c in range(3)]
        c = int(np.argmax(keys))
        u = O.uniform(6, j, 3, O.P_RESID_INCHUNK, 0)
        k = int(np.searchsorted(np.cumsum(special.softmax(lw[4 * c:4 * c + 4])), u, side="right"))
        assert x == 4 * c + k and np.isfinite(lw[x])
        assert abs(lse - special.logsumexp(lw)) < 1e-12


def _chi2_p(counts, probs):
    exp = probs * counts.sum()
    return stats.chisquare(counts, exp).pvalue


@pytest.mark.parametrize("T", [0.7, 1.0])
@pytest.mark.parametrize("CS,variant", [(1, 0), (2, 0), (3, 0), (8, 0), (8, 1), (1, 2), (2, 2), (3, 2), (8, 2)])
def test_samplers_chi_square(T, CS, variant):
    rng = np.random.default_rng(10)
    z = rng.normal(0, 1.2, 8)
    lw = z / T
    counts = O.trials_sampler(lw, 1234 + 7 * CS + (5, 8, 0)[variant], 1_000_000, variant, CS=CS)
    assert _chi2_p(counts, special.softmax(lw)) > 1e-3


def test_chi_square_detects_a_wrong_law():
    # the same test must reject a sampler drawing from a slightly different law
    rng = np.random.default_rng(10)
    lw = rng.normal(0, 1.2, 8)
    wrong = special.softmax(lw * 1.02)
    for variant in (0, 2):
        counts = O.trials_sampler(lw, 77, 1_000_000, variant, CS=2)
        assert _chi2_p(counts, wrong) < 1e-6


def test_sample_request_greedy_chain():
    rng = np.random.default_rng(5)
    B, gamma, V, r = 2, 4, 64, 3
    base = rng.normal(0, 2, (B, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.7, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.7, (V, r)).astype(np.float32)
    anchor = np.array([5, 17], np.int32)
    for j in range(B):
        tok, lse, zx, mg = O.sample_request(base, W1, W2, anchor[j], j, 0.0, 0, 1024)
        prev = anchor[j]
        for i in range(gamma):
            z = base[j, i].astype(np.float64) + W2.astype(np.float64) @ W1[prev].astype(np.float64)
            assert tok[i] == int(np.argmax(z))
            assert np.isnan(lse[i])
            assert abs(zx[i] - z[tok[i]]) < 1e-12
            prev = tok[i]


def test_block_logits_with_the_drafts_own_tokens_replays_the_draft():
    # teacher forcing with the greedy draft's own tokens must give back, at every position, the
    # draft's argmax and its z at the token (the previous-token rule against the sampler's carry)
    rng = np.random.default_rng(8)
    B, gamma, V, r = 3, 5, 96, 4
    base = rng.normal(0, 2, (B, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.7, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.7, (V, r)).astype(np.float32)
    anchor = np.array([5, 17, 95], np.int32)
    toks = np.zeros((B, gamma), np.int32)
    zats = np.zeros((B, gamma))
    for j in range(B):
        tok, _, zx, _ = O.sample_request(base, W1, W2, anchor[j], j, 0.0, 0, 1024)
        toks[j], zats[j] = tok, zx
    z = O.block_logits(base, W1, W2, anchor, toks)
    assert z.shape == (B, gamma, V)
    for j in range(B):
        for i in range(gamma):
            assert int(np.argmax(z[j, i])) == toks[j, i]
            assert z[j, i, toks[j, i]] == zats[j, i]
    # a different token at position i changes only position i + 1's bias
    t2 = toks.copy()
    t2[1, 2] = (t2[1, 2] + 1) % V
    z2 = O.block_logits(base, W1, W2, anchor, t2)
    changed = np.argwhere(np.any(z2 != z, axis=-1))
    assert changed.tolist() == [[1, 3]]
    # no Markov head: z is the base row
    assert np.array_equal(O.block_logits(base, None, None, anchor, toks), base.astype(np.float64))


def test_sample_request_carries_token_and_lse():
    rng = np.random.default_rng(6)
    B, gamma, V, r = 1, 5, 50, 4
    base = rng.normal(0, 1, (B, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 1.0, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 1.0, (V, r)).astype(np.float32)
    T = 0.8
    tok, lse, zx, mg = O.sample_request(base, W1, W2, 7, 0, T, 99, 16, CS=4)
    prev = 7
    for i in range(gamma):
        z = base[0, i].astype(np.float64) + W2.astype(np.float64) @ W1[prev].astype(np.float64)
        x, m, l = O.chunk_gumbel(z / T, 99, 0, i + 1, CS=4)
        assert tok[i] == x and abs(lse[i] - special.logsumexp(z / T)) < 1e-12
        assert abs(zx[i] - z[x]) < 1e-12
        prev = x


# ---------------------------------------------------------------- final-logit softcap (page "03 · DSpark 建模", 3.12)
def test_softcap_limits_and_bounds():
    rng = np.random.default_rng(5)
    V, r = 64, 4
    base = (rng.normal(0, 20, V)).astype(np.float32)
    W1 = rng.normal(0, 1.0, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 1.0, (V, r)).astype(np.float32)
    prev = 7
    plain = O.markov_logits(base, W1, W2, prev)
    bias = plain - base.astype(np.float64)
    # a cap far above every logit leaves them unchanged
    assert np.allclose(O.markov_logits(base, W1, W2, prev, softcap=1e30), plain, rtol=1e-15, atol=0)
    for s in (0.5, 3.0, 30.0):
        capped = O.markov_logits(base, None, None, 0, softcap=s)  # rank 0: the capped base alone
        assert np.all(np.abs(capped) <= s)  # (tanh reaches 1 in double for large arguments)
        order = np.argsort(base, kind="stable")
        assert np.all(np.diff(capped[order]) >= 0)  # monotone in the base logit
        neg = O.markov_logits(-base, None, None, 0, softcap=s)
        assert np.array_equal(neg, -capped)  # odd
        # the bias is added after the cap: with the Markov head the difference is the bias itself
        assert np.allclose(O.markov_logits(base, W1, W2, prev, softcap=s) - capped, bias, rtol=0, atol=1e-12)
    # with the bias added after the cap, z itself leaves [-s, s] when the bias is large
    z = O.markov_logits(base, W1, W2, prev, softcap=0.5)
    assert np.abs(z).max() > 0.5
    # closed form: base = s atanh(q) is capped to s q
    s = 4.0
    q = np.array([-0.9, -0.25, 0.0, 0.25, 0.5, 0.9])
    b = (s * np.arctanh(q)).astype(np.float32)
    got = O.markov_logits(b, None, None, 0, softcap=s)
    want = s * np.tanh(np.arctanh(q) + (b.astype(np.float64) / s - np.arctanh(q)))  # exact for the rounded b
    assert np.allclose(got, want, rtol=0, atol=1e-12) and np.allclose(got, s * q, rtol=0, atol=1e-6)


def test_softcap_greedy_draft_is_the_capped_argmax():
    rng = np.random.default_rng(9)
    B, g, V, r = 1, 3, 300, 4
    base = rng.normal(0, 5, (B, g, V)).astype(np.float32)
    base[0, :, 17] = 40.0  # towers over the rest uncapped ...
    base[0, :, 200] = 39.0
    W1 = rng.normal(0, 0.01, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.01, (V, r)).astype(np.float32)
    W1[3] = [1.0, 0.0, 0.0, 0.0]  # the anchor's row: bias_v = W2[v, 0] at position 1
    W2[17, 0], W2[200, 0] = 0.0, 0.5  # ... while a cap of 2 flattens the top and the bias then decides
    tok, lse, zx, mg = O.sample_request(base, W1, W2, 3, 0, 0.0, 0, 64, softcap=2.0)
    prev = 3
    for i in range(g):
        z = O.markov_logits(base[0, i], W1, W2, prev, softcap=2.0)
        assert tok[i] == int(np.argmax(z)) and zx[i] == z[tok[i]]
        prev = int(tok[i])
    assert tok[0] == 200  # capped: 2 tanh(19.5) + 0.5 > 2 tanh(20)
    tok0, *_ = O.sample_request(base, W1, W2, 3, 0, 0.0, 0, 64)
    assert tok0[0] == 17  # without the cap the tower wins: 40 > 39 + 0.5
