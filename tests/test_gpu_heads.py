"""Parity of the Gated and RNN Markov heads (dspark_markov_sample_block_head, dspark_verify_head)
with the oracle (page "03 · DSpark 建模：Markov 与 Confidence", section 3.7).  Inputs of the
verify test (drafted tokens, LSE, logits, head vectors) come from the oracle's head sampler.

Head-vector tolerance: every component of u is a fp32 dot product of n = r + d (gated) or 2r + d
(rnn) terms followed by sigmoid / tanh (slopes at most 1/4 and 1); the rounding of such a sum is
below n 2^-24 sum |w z|, which for the weights drawn here (std 0.2, inputs of order 1, n <= 320)
stays under 1e-4 in the worst case and is near 1e-6 in practice.  The test uses 2e-5 absolute +
1e-5 relative and the RNN state, being a convex mix of bounded terms, does not amplify it."""
import numpy as np
import pytest
import torch

import oracle as O
from parity import MARGIN, Tally, close, compare_block
from semi_ar_draft_gb300 import api, binding
from semi_ar_draft_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TS = 1024
KINDS = {"gated": W.HEAD_GATED, "rnn": W.HEAD_RNN}


def head_case(name, B, gamma, V, r, d, T, kind, *, ldt=torch.float32, wdt=torch.float32, w_std=0.3,
              hw_std=0.2, data_seed=0):
    wl = W.make_sample_workload(name, B, gamma, V, r, T, device="cuda", data_seed=data_seed, philox_seed=13,
                                logits_dtype=ldt, w_dtype=wdt, w_std=w_std, base_std=2.0)
    h = W.make_head_inputs(wl, kind, d, data_seed=data_seed, w_std=hw_std)
    return wl, h


def run_head(wl, h, kind, softcap=0.0):
    t = wl.tensors
    return api.markov_sample_block_head(t["base"], t["W1"], t["W2"], t["anchor"], wl.T, wl.seed, kind, h["hidden"],
                                        h["Wg"], h.get("Wc"), h.get("Wo"), softcap=softcap)


def oracle_head(wl, h, kind, j, softcap=0.0):
    t = wl.tensors
    nv = W.np_view
    return O.sample_request_head(nv(t["base"]), nv(t["W1"]), nv(t["W2"]), int(t["anchor"][j]), j, wl.T, wl.seed, TS,
                                 kind, nv(h["hidden"]), nv(h["Wg"]), nv(h["Wc"]) if "Wc" in h else None,
                                 nv(h["Wo"]) if "Wo" in h else None, softcap=softcap)


def compare(wl, h, kind, requests=None, softcap=0.0):
    tok, lse, zat, u, ws = run_head(wl, h, kind, softcap)
    torch.cuda.synchronize()
    assert binding.dspark_get_device_status(ws) == 0
    g_tok, g_lse, g_zat, g_u = (x.cpu().numpy() for x in (tok, lse, zat, u))
    tally = Tally()
    for j in (range(wl.B) if requests is None else requests):
        rt, rl, rz, rm, ru = oracle_head(wl, h, kind, j, softcap)
        n = compare_block(tally, g_tok[j], g_lse[j], g_zat[j], (rt, rl, rz, rm), wl.T, j)
        # u of position i depends on the drafted tokens before it: compare while they agree
        close(g_u[j, : n + (n < wl.gamma)], ru[: n + (n < wl.gamma)], rtol=1e-5, atol=2e-5, what=f"u j={j}")
    tally.check_fraction()
    return g_tok, g_u


@pytest.mark.parametrize("kind", ["gated", "rnn"])
@pytest.mark.parametrize("T", [0.0, 1.0])
def test_small_fp32_ragged(kind, T):
    # V = 3000: two full tiles and a ragged one; B = 19: a full and a partial row block of 16
    wl, h = head_case("hs", 19, 5, 3000, 16, 24, T, KINDS[kind], data_seed=1)
    compare(wl, h, KINDS[kind])


@pytest.mark.parametrize("kind", ["gated", "rnn"])
def test_bf16_mixed_ranks(kind):
    wl, h = head_case("hb", 7, 4, 5000, 64, 96, 0.8, KINDS[kind], ldt=torch.bfloat16, wdt=torch.bfloat16,
                      w_std=0.15, data_seed=2)
    compare(wl, h, KINDS[kind])


@pytest.mark.parametrize("kind", ["gated", "rnn"])
def test_full_vocab_b32_r64_sampled_requests(kind):
    # the b32 shape (V = 151936, r = 64, bf16) with a hidden size of 256
    wl, h = head_case("h32", 32, 8, W.VOCAB, 64, 256, 1.0, KINDS[kind], ldt=torch.bfloat16, wdt=torch.bfloat16,
                      w_std=0.1, data_seed=3)
    compare(wl, h, KINDS[kind], requests=[0, 15, 16, 31])


def test_head_changes_the_draft_and_softcap():
    # the head's bias moves the drafted tokens away from the vanilla head's; a softcap still applies
    wl, h = head_case("hc", 16, 4, 4096, 32, 32, 0.0, W.HEAD_RNN, w_std=0.6, hw_std=0.5, data_seed=4)
    t = wl.tensors
    g_tok, _ = compare(wl, h, W.HEAD_RNN)
    van = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], 0.0, wl.seed)[0].cpu().numpy()
    assert (g_tok != van).mean() > 0.2
    compare(wl, h, W.HEAD_RNN, softcap=2.5)


def test_gated_zero_weights_is_half_gate_vanilla():
    # Wg = 0: gate 1/2 exactly, so the drafted tokens are those of the vanilla head with W1 / 2
    wl, h = head_case("hz", 12, 4, 2048, 16, 8, 1.0, W.HEAD_GATED, data_seed=5)
    h["Wg"].zero_()
    t = wl.tensors
    tok, lse, zat, u, _ = run_head(wl, h, W.HEAD_GATED)
    ref = api.markov_sample_block(t["base"], t["W1"] * 0.5, t["W2"], t["anchor"], wl.T, wl.seed)
    torch.cuda.synchronize()
    assert torch.equal(tok, ref[0])
    close(lse.cpu().numpy(), ref[1].cpu().numpy(), rtol=1e-6, atol=1e-6, what="lse")


@pytest.mark.parametrize("kind", ["gated", "rnn"])
def test_verify_head(kind):
    wl, h = head_case("hv", 13, 4, 3000, 16, 20, 1.0, KINDS[kind], data_seed=6)
    t = wl.tensors
    nv = W.np_view
    base, W2, target = nv(t["base"]), nv(t["W2"]), nv(t["target"])
    anchor = t["anchor"].cpu().numpy()
    B, g, r = wl.B, wl.gamma, wl.r
    tok = np.zeros((B, g), np.int32)
    lse = np.zeros((B, g), np.float32)
    zat = np.zeros((B, g), np.float32)
    u = np.zeros((B, g, r), np.float32)
    for j in range(B):
        rt, rl, rz, _, ru = oracle_head(wl, h, KINDS[kind], j)
        tok[j], lse[j], zat[j], u[j] = rt, rl, rz, ru
    dev = "cuda"
    n, corr, ws = api.verify_head(t["base"], torch.from_numpy(u).to(dev), t["W2"], t["anchor"],
                                  torch.from_numpy(tok).to(dev), torch.from_numpy(lse).to(dev),
                                  torch.from_numpy(zat).to(dev), t["target"], wl.T, wl.seed)
    torch.cuda.synchronize()
    assert binding.dspark_get_device_status(ws) == 0
    n, corr = n.cpu().numpy(), corr.cpu().numpy()
    tally = Tally()
    for j in range(B):
        rn, rc, rm, _ = O.verify_request(base, nv(t["W1"]), W2, int(anchor[j]), j, tok[j], lse[j], zat[j], target, g,
                                         wl.T, wl.seed, TS, head_vec=u[j])
        tally.total += 1
        if (n[j], corr[j]) != (rn, rc):
            assert rm < MARGIN, f"request {j}: gpu ({n[j]}, {corr[j]}) vs oracle ({rn}, {rc}) margin {rm}"
            tally.excluded += 1
    tally.check_fraction()
    assert (n < g).any()  # residual draws from the head's q were exercised


def test_rnn_state_does_not_fit_is_unsupported():
    # B r floats x 3 of RNN state beyond one block's shared memory
    wl, h = head_case("hu", 512, 1, 1024, 64, 8, 1.0, W.HEAD_RNN, data_seed=7)
    with pytest.raises(binding.DsparkError) as e:
        run_head(wl, h, W.HEAD_RNN)
    assert e.value.status == 2
