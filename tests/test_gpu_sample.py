"""Parity of dspark_markov_sample_block (CUDA) with the oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle as O
from parity import Tally, close, compare_block
from semi_ar_draft_gb300 import api, binding
from semi_ar_draft_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TS = 1024


def run_and_compare(wl, requests=None, tally=None, softcap=0.0):
    t = wl.tensors
    tok, lse, zat, ws = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], wl.T, wl.seed,
                                                softcap=softcap)
    torch.cuda.synchronize()
    assert binding.dspark_get_device_status(ws) == 0
    base = W.np_view(t["base"])
    W1 = None if t["W1"] is None else W.np_view(t["W1"])
    W2 = None if t["W2"] is None else W.np_view(t["W2"])
    anchor = t["anchor"].cpu().numpy()
    g_tok, g_lse, g_zat = tok.cpu().numpy(), lse.cpu().numpy(), zat.cpu().numpy()
    tally = tally or Tally()
    reqs = range(wl.B) if requests is None else requests
    for j in reqs:
        ref = O.sample_request(base, W1, W2, int(anchor[j]), int(j), wl.T, wl.seed, TS, softcap=softcap)
        compare_block(tally, g_tok[j], g_lse[j], g_zat[j], ref, wl.T, j)
    return tally, (tok, lse, zat)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tiny_fp32(T):
    wl = W.tiny(T, device="cuda")
    tally, _ = run_and_compare(wl)
    tally.check_fraction()


@pytest.mark.parametrize("r", [0, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("T", [0.0, 0.8])
def test_bf16_ranks_ragged(r, T):
    # V = 5000: four full tiles and a ragged one; B = 20: a full and a partial row block
    wl = W.make_sample_workload("ragged", 20, 3, 5000, r, T, device="cuda", data_seed=r + 7, philox_seed=11,
                                planted=3)
    tally, _ = run_and_compare(wl)
    tally.check_fraction()


@pytest.mark.parametrize("wdt,r", [(torch.float32, 16), (torch.float32, 24), (torch.bfloat16, 24)])
def test_cuda_core_path(wdt, r):
    wl = W.make_sample_workload("gemv", 5, 4, 3000, r, 1.0, device="cuda", data_seed=3, philox_seed=5,
                                logits_dtype=torch.float32, w_dtype=wdt, w_std=0.3)
    tally, _ = run_and_compare(wl)
    tally.check_fraction()


def test_unaligned_vocab_scalar_loads():
    wl = W.make_sample_workload("odd", 3, 3, 1001, 32, 1.0, device="cuda", data_seed=9, philox_seed=2, w_std=0.3)
    tally, _ = run_and_compare(wl)
    tally.check_fraction()


def test_fp32_logits_bf16_weights_single_step():
    wl = W.make_sample_workload("f32b", 17, 1, 2048, 64, 0.5, device="cuda", data_seed=4, philox_seed=9,
                                logits_dtype=torch.float32, w_std=0.2)
    tally, _ = run_and_compare(wl)
    tally.check_fraction()


def test_markov_bias_matters():
    # with large weights the bias changes the drafted tokens: parity then really checks the GEMM
    wl = W.make_sample_workload("bias", 16, 4, 4096, 64, 0.0, device="cuda", data_seed=1, w_std=0.5)
    tally, (tok, _, _) = run_and_compare(wl)
    t = wl.tensors
    no_bias = torch.argmax(t["base"].float(), dim=-1).to(torch.int32)
    assert (tok != no_bias).float().mean().item() > 0.5


def test_deterministic_and_seed_dependent():
    wl = W.make_sample_workload("det", 8, 4, 3000, 64, 1.0, device="cuda", data_seed=2)
    t = wl.tensors
    a = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], 1.0, 5)[0].clone()
    b = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], 1.0, 5)[0].clone()
    c = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], 1.0, 6)[0].clone()
    assert torch.equal(a, b) and not torch.equal(a, c)


def test_anchor_out_of_range_sets_status():
    wl = W.make_sample_workload("bad", 4, 2, 2048, 16, 1.0, device="cuda")
    t = wl.tensors
    anchor = t["anchor"].clone()
    anchor[2] = 5000
    _, _, _, ws = api.markov_sample_block(t["base"], t["W1"], t["W2"], anchor, 1.0, 0)
    assert binding.dspark_get_device_status(ws) == 7


def test_full_b32_r64():
    wl = W.b32_r64(device="cuda")
    tally, _ = run_and_compare(wl)
    tally.check_fraction()


def test_full_b128_r256_sampled_requests():
    # the tensor-core sampler at rank 256: first and last lanes of each 32-lane TMEM quarter
    wl = W.b128_r256(device="cuda")
    tally, _ = run_and_compare(wl, requests=[0, 31, 32, 45, 63, 64, 96, 127])
    tally.check_fraction()


def test_full_b512_r64_sampled_requests():
    # the tensor-core sampler: requests from every 128-request row block, first and last lanes
    wl = W.b512_sched(device="cuda")
    tally, _ = run_and_compare(wl, requests=[0, 1, 31, 32, 127, 128, 200, 255, 256, 300, 383, 384, 450, 510, 511])
    tally.check_fraction()


# ---------------------------------------------------------------- tensor-core sampler (B >= 64, r = 64)
@pytest.mark.parametrize("T", [0.0, 0.8])
def test_tc_ragged_vocab_and_row_block(T):
    # V = 5000: four full 1024-id tiles and a ragged one whose last 64-id copy is partly past V;
    # B = 200: one full 128-request row block and a partial one
    wl = W.make_sample_workload("tc", 200, 3, 5000, 64, T, device="cuda", data_seed=31, philox_seed=4, planted=3,
                                w_std=0.3)
    tally, _ = run_and_compare(wl)
    tally.check_fraction()


@pytest.mark.parametrize("B,gamma,V,T", [(64, 2, 2048, 0.7), (300, 5, 4096, 1.0), (128, 6, 3000, 0.0),
                                         (129, 4, 1032, 1.3)])
def test_tc_shapes(B, gamma, V, T):
    wl = W.make_sample_workload("tcs", B, gamma, V, 64, T, device="cuda", data_seed=B + V, philox_seed=B,
                                planted=2, w_std=0.4)
    tally, _ = run_and_compare(wl)
    tally.check_fraction()


@pytest.mark.parametrize("r", [128, 256])
@pytest.mark.parametrize("B,gamma,V,T", [(200, 3, 5000, 0.8), (128, 4, 3000, 0.0), (64, 2, 2048, 1.3)])
def test_tc_higher_ranks(r, B, gamma, V, T):
    # ranks 128 and 256: K-chunked operands, two ring stages per accumulator (N = 64); ragged
    # vocabularies and a partial row block
    wl = W.make_sample_workload("tcr", B, gamma, V, r, T, device="cuda", data_seed=r + B, philox_seed=7, planted=2,
                                w_std=0.25)
    tally, _ = run_and_compare(wl)
    tally.check_fraction()


def test_tc_rank256_bias_matters():
    wl = W.make_sample_workload("tcb256", 128, 3, 4096, 256, 0.0, device="cuda", data_seed=9, w_std=0.3)
    tally, (tok, _, _) = run_and_compare(wl)
    no_bias = torch.argmax(wl.tensors["base"].float(), dim=-1).to(torch.int32)
    assert (tok != no_bias).float().mean().item() > 0.5


def test_tc_bias_matters_and_deterministic():
    wl = W.make_sample_workload("tcb", 128, 4, 4096, 64, 0.0, device="cuda", data_seed=8, w_std=0.5)
    tally, (tok, _, _) = run_and_compare(wl)
    t = wl.tensors
    no_bias = torch.argmax(t["base"].float(), dim=-1).to(torch.int32)
    assert (tok != no_bias).float().mean().item() > 0.5
    wl = W.make_sample_workload("tcd", 160, 4, 3000, 64, 1.0, device="cuda", data_seed=2)
    t = wl.tensors
    a = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], 1.0, 5)[0].clone()
    b = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], 1.0, 5)[0].clone()
    c = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], 1.0, 6)[0].clone()
    assert torch.equal(a, b) and not torch.equal(a, c)


def test_tc_anchor_out_of_range_sets_status():
    wl = W.make_sample_workload("tcbad", 96, 2, 2048, 64, 1.0, device="cuda")
    t = wl.tensors
    anchor = t["anchor"].clone()
    anchor[70] = 5000
    _, _, _, ws = api.markov_sample_block(t["base"], t["W1"], t["W2"], anchor, 1.0, 0)
    assert binding.dspark_get_device_status(ws) == 7


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_vocabulary_beyond_one_tile_per_sm(T):
    # 160000 ids = 157 tiles: more tiles than SMs, so blocks own several tiles (no shared-memory staging)
    wl = W.make_sample_workload("wide", 4, 2, 160000, 64, T, device="cuda", data_seed=12, philox_seed=3, planted=2)
    tally, _ = run_and_compare(wl)
    tally.check_fraction()


# ---------------------------------------------------------------- teacher-forced block logits
def _block_logits_check(wl, tokens):
    t = wl.tensors
    z, ws = api.markov_block_logits(t["base"], t["W1"], t["W2"], t["anchor"], tokens)
    torch.cuda.synchronize()
    assert binding.dspark_get_device_status(ws) == 0
    base = W.np_view(t["base"])
    W1 = None if t["W1"] is None else W.np_view(t["W1"])
    W2 = None if t["W2"] is None else W.np_view(t["W2"])
    anchor, toks = t["anchor"].cpu().numpy(), tokens.cpu().numpy()
    ref = O.block_logits(base, W1, W2, anchor, toks)
    # Tolerance from the arithmetic: the kernel adds r products (bf16 or fp32 operands, exact in
    # fp32) in fp32, so its error scales with the summed magnitude S = |base| + sum_k |W2[v,k] W1[prev,k]|
    # (about sqrt(r) 2^-24 S, at most 1e-6 S for r <= 256), not with |z|, which cancellation can
    # make small.  Plus the usual 1e-5 relative term.
    S = np.abs(base.astype(np.float64))
    if W1 is not None:
        prev = np.concatenate([anchor[:, None], toks[:, :-1]], axis=1).astype(np.int64)
        aW1 = np.abs(W1.astype(np.float64))[prev]  # [B, gamma, r]
        S = S + np.einsum("bgk,vk->bgv", aW1, np.abs(W2.astype(np.float64)))
    got = z.cpu().numpy().astype(np.float64)
    bad = np.abs(got - ref) > 1e-5 * np.abs(ref) + 1e-6 * S
    assert not bad.any(), f"block logits: {int(bad.sum())} values off; first {got[bad][:5]} vs {ref[bad][:5]}"


@pytest.mark.parametrize("B,gamma,V,r", [(3, 5, 5000, 64), (2, 7, 4096, 16), (1, 3, 2048, 256), (32, 8, 151936, 64)])
def test_block_logits_tensor_core(B, gamma, V, r):
    wl = W.make_sample_workload("blk", B, gamma, V, r, 1.0, device="cuda", data_seed=B * 10 + r, w_std=0.3)
    g = torch.Generator(device="cpu").manual_seed(B + gamma)
    tokens = torch.randint(0, V, (B, gamma), generator=g, dtype=torch.int32).cuda()
    _block_logits_check(wl, tokens)


@pytest.mark.parametrize("wdt,r", [(torch.float32, 24), (torch.bfloat16, 24), (torch.float32, 0)])
def test_block_logits_cuda_core(wdt, r):
    wl = W.make_sample_workload("blkc", 4, 4, 3001, r, 1.0, device="cuda", data_seed=5, logits_dtype=torch.float32,
                                w_dtype=wdt, w_std=0.3)
    tokens = torch.randint(0, 3001, (4, 4), dtype=torch.int32).cuda()
    _block_logits_check(wl, tokens)


def test_block_logits_token_out_of_range_sets_status():
    wl = W.make_sample_workload("blkbad", 2, 3, 2048, 16, 1.0, device="cuda")
    t = wl.tensors
    tokens = torch.tensor([[1, 5000, 3], [4, 5, 6]], dtype=torch.int32, device="cuda")
    _, ws = api.markov_block_logits(t["base"], t["W1"], t["W2"], t["anchor"], tokens)
    assert binding.dspark_get_device_status(ws) == 7  # DSPARK_ERR_TOKEN_RANGE


# ---------------------------------------------------------------- final-logit softcap (page "03 · DSpark 建模", 3.12)
@pytest.mark.parametrize("T", [0.0, 1.0])
@pytest.mark.parametrize("B,logits_dtype", [(20, torch.bfloat16), (96, torch.bfloat16), (5, torch.float32)])
def test_softcap(T, B, logits_dtype):
    # staged sampler (bf16, 20 requests), the 96-request case (eligible for the tensor-core sampler
    # without a cap, so it shows the cap routes elsewhere) and the general fp32 kernel; cap 4 against
    # base logits ~N(0, 3) with planted peaks of +8: most of the mass sits where the cap bends
    wl = W.make_sample_workload("cap", B, 3, 5000, 64, T, device="cuda", data_seed=B + 3, philox_seed=7, planted=3,
                                logits_dtype=logits_dtype, w_std=0.3)
    tally, _ = run_and_compare(wl, softcap=4.0)
    tally.check_fraction()


def test_softcap_block_logits():
    wl = W.make_sample_workload("capb", 3, 4, 3000, 64, 1.0, device="cuda", data_seed=11, w_std=0.3)
    t = wl.tensors
    tokens = torch.randint(0, 3000, (3, 4), dtype=torch.int32).cuda()
    z, ws = api.markov_block_logits(t["base"], t["W1"], t["W2"], t["anchor"], tokens, softcap=2.5)
    torch.cuda.synchronize()
    assert binding.dspark_get_device_status(ws) == 0
    ref = O.block_logits(W.np_view(t["base"]), W.np_view(t["W1"]), W.np_view(t["W2"]), t["anchor"].cpu().numpy(),
                         tokens.cpu().numpy(), softcap=2.5)
    close(z.cpu().numpy(), ref, rtol=1e-5, atol=2e-6, what="capped block logits")


def test_softcap_rejects_bad_values():
    wl = W.make_sample_workload("capbad", 2, 2, 1024, 16, 1.0, device="cuda")
    t = wl.tensors
    for bad in (-1.0, float("inf"), float("nan")):
        with pytest.raises(binding.DsparkError) as e:
            api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], 1.0, 0, softcap=bad)
        assert e.value.status == 1
