"""Parity of dspark_verify (CUDA) with the oracle.  Inputs of the verify-only tests (drafted
tokens, their LSE and logits) come from the oracle's sampler, never from the CUDA path."""
import numpy as np
import pytest
import torch

import oracle as O
from parity import MARGIN, Tally, compare_block
from semi_ar_draft_gb300 import api, binding
from semi_ar_draft_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TS = 1024


def host(wl):
    t = wl.tensors
    return (W.np_view(t["base"]), None if t["W1"] is None else W.np_view(t["W1"]),
            None if t["W2"] is None else W.np_view(t["W2"]), t["anchor"].cpu().numpy(), W.np_view(t["target"]))


def oracle_drafts(wl, softcap=0.0):
    base, W1, W2, anchor, _ = host(wl)
    B, g = wl.B, wl.gamma
    tok = np.zeros((B, g), np.int32)
    lse = np.zeros((B, g), np.float32)
    zat = np.zeros((B, g), np.float32)
    for j in range(B):
        rt, rl, rz, _ = O.sample_request(base, W1, W2, int(anchor[j]), j, wl.T, wl.seed, TS, softcap=softcap)
        tok[j], lse[j], zat[j] = rt, rl.astype(np.float32), rz.astype(np.float32)
    return tok, lse, zat


def verify_both(wl, tok, lse, zat, vlen=None, csr=False, softcap=0.0):
    t = wl.tensors
    base, W1, W2, anchor, target = host(wl)
    dev = "cuda"
    gt_tok = torch.from_numpy(tok).to(dev)
    gt_lse = torch.from_numpy(lse).to(dev)
    gt_zat = torch.from_numpy(zat).to(dev)
    vl = None if vlen is None else torch.from_numpy(vlen.astype(np.int32)).to(dev)
    if csr:
        # flattened target rows: request j owns L_j + 1 rows (its verified rows and the bonus row)
        L = vlen if vlen is not None else np.full(wl.B, wl.gamma)
        nrows = np.minimum(L + 1, wl.gamma_t)
        off = np.concatenate([[0], np.cumsum(nrows)]).astype(np.int32)
        idx = np.concatenate([j * wl.gamma_t + np.arange(nrows[j]) for j in range(wl.B)])
        flat = t["target"].reshape(wl.B * wl.gamma_t, wl.V)[torch.from_numpy(idx).to(dev)].contiguous()
        n, corr, ws = api.verify(t["base"], t["W1"], t["W2"], t["anchor"], gt_tok, gt_lse, gt_zat, flat, wl.T,
                                 wl.seed, verify_len=vl, target_row_offsets=torch.from_numpy(off).to(dev))
    else:
        n, corr, ws = api.verify(t["base"], t["W1"], t["W2"], t["anchor"], gt_tok, gt_lse, gt_zat, t["target"],
                                 wl.T, wl.seed, verify_len=vl, softcap=softcap)
    torch.cuda.synchronize()
    assert binding.dspark_get_device_status(ws) == 0
    n, corr = n.cpu().numpy(), corr.cpu().numpy()
    tally = Tally()
    for j in range(wl.B):
        Lj = wl.gamma if vlen is None else int(vlen[j])
        tgt = target if not csr else target[:, : wl.gamma_t]
        rn, rc, rm, _ = O.verify_request(base, W1, W2, int(anchor[j]), j, tok[j], lse[j], zat[j], tgt, Lj, wl.T,
                                         wl.seed, TS, softcap=softcap)
        tally.total += 1
        if (n[j], corr[j]) != (rn, rc):
            assert rm < MARGIN, f"request {j}: gpu (n={n[j]}, corr={corr[j]}) vs oracle ({rn}, {rc}) margin {rm}"
            tally.excluded += 1
    tally.check_fraction()
    return n, corr


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tiny(T):
    wl = W.tiny(T, device="cuda")
    verify_both(wl, *oracle_drafts(wl))


@pytest.mark.parametrize("r,T", [(64, 1.0), (64, 0.0), (0, 0.7), (256, 0.7), (16, 1.3)])
def test_ragged_dense(r, T):
    wl = W.make_sample_workload("v", 21, 4, 5000, r, T, device="cuda", data_seed=r + 1, philox_seed=3,
                                target_sigma=0.7, planted=2)
    n, corr = verify_both(wl, *oracle_drafts(wl))
    assert (n < wl.gamma).any()  # some rejections exercised the residual path


def test_bonus_rows_and_verify_len():
    wl = W.make_sample_workload("vb", 19, 5, 3000, 64, 1.0, device="cuda", data_seed=5, target_sigma=0.1, gamma_t=6)
    tok, lse, zat = oracle_drafts(wl)
    vlen = np.random.default_rng(0).integers(1, 6, wl.B)
    n, corr = verify_both(wl, tok, lse, zat, vlen=vlen)
    assert (n == vlen).any() and (corr >= 0).all()  # all-accepted requests drew a bonus token


def test_flattened_target_rows():
    wl = W.make_sample_workload("vf", 18, 5, 3000, 32, 0.9, device="cuda", data_seed=6, target_sigma=0.3, gamma_t=6)
    tok, lse, zat = oracle_drafts(wl)
    vlen = np.random.default_rng(1).integers(1, 6, wl.B)
    verify_both(wl, tok, lse, zat, vlen=vlen, csr=True)


def test_greedy_bonus():
    wl = W.make_sample_workload("vg", 9, 3, 2048, 64, 0.0, device="cuda", data_seed=8, target_sigma=0.01, gamma_t=4)
    tok, lse, zat = oracle_drafts(wl)
    n, corr = verify_both(wl, tok, lse, zat)
    assert (n == 3).any()


def test_bad_token_sets_status():
    wl = W.make_sample_workload("vt", 4, 2, 2048, 16, 1.0, device="cuda")
    tok, lse, zat = oracle_drafts(wl)
    tok[1, 0] = -3
    t = wl.tensors
    _, _, ws = api.verify(t["base"], t["W1"], t["W2"], t["anchor"], torch.from_numpy(tok).cuda(),
                          torch.from_numpy(lse).cuda(), torch.from_numpy(zat).cuda(), t["target"], 1.0, 0)
    assert binding.dspark_get_device_status(ws) == 7


def end_to_end(wl, requests):
    t = wl.tensors
    base, W1, W2, anchor, target = host(wl)
    tok, lse, zat, _ = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], wl.T, wl.seed)
    n, corr, ws = api.verify(t["base"], t["W1"], t["W2"], t["anchor"], tok, lse, zat, t["target"], wl.T, wl.seed)
    torch.cuda.synchronize()
    g_tok, g_lse, g_zat = tok.cpu().numpy(), lse.cpu().numpy(), zat.cpu().numpy()
    n, corr = n.cpu().numpy(), corr.cpu().numpy()
    tally = Tally()
    for j in requests:
        ref = O.sample_request(base, W1, W2, int(anchor[j]), j, wl.T, wl.seed, TS)
        agree = compare_block(tally, g_tok[j], g_lse[j], g_zat[j], ref, wl.T, j)
        if agree < wl.gamma:
            continue  # an excluded draft decision: the downstream verify is not comparable
        rn, rc, rm, _ = O.verify_request(base, W1, W2, int(anchor[j]), j, ref[0], ref[1].astype(np.float32),
                                         ref[2].astype(np.float32), target, wl.gamma, wl.T, wl.seed, TS)
        tally.total += 1
        if (n[j], corr[j]) != (rn, rc):
            assert rm < MARGIN, f"request {j}: ({n[j]}, {corr[j]}) vs ({rn}, {rc}) margin {rm}"
            tally.excluded += 1
    tally.check_fraction()


def test_end_to_end_b32_r64():
    end_to_end(W.b32_r64(device="cuda"), range(32))


def test_end_to_end_b128_r256_sampled():
    end_to_end(W.b128_r256(device="cuda"), [3, 64, 126])


def test_end_to_end_b512_scheduled_lengths_sampled():
    # the b512 configuration as the bench runs it: lengths from the scheduler, then sample and verify
    wl = W.b512_sched(device="cuda")
    t = wl.tensors
    L, _, _, _ = api.schedule_verify_len(t["conf"], wl.budget)
    base, W1, W2, anchor, target = host(wl)
    tok, lse, zat, _ = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], wl.T, wl.seed)
    n, corr, ws = api.verify(t["base"], t["W1"], t["W2"], t["anchor"], tok, lse, zat, t["target"], wl.T, wl.seed,
                             verify_len=L)
    torch.cuda.synchronize()
    assert binding.dspark_get_device_status(ws) == 0
    L = L.cpu().numpy()
    assert L.sum() <= wl.budget and L.min() >= 1
    g_tok, g_lse, g_zat = tok.cpu().numpy(), lse.cpu().numpy(), zat.cpu().numpy()
    n, corr = n.cpu().numpy(), corr.cpu().numpy()
    tally = Tally()
    for j in (0, 137, 300, 511):
        ref = O.sample_request(base, W1, W2, int(anchor[j]), j, wl.T, wl.seed, TS)
        if compare_block(tally, g_tok[j], g_lse[j], g_zat[j], ref, wl.T, j) < wl.gamma:
            continue
        rn, rc, rm, _ = O.verify_request(base, W1, W2, int(anchor[j]), j, ref[0], ref[1].astype(np.float32),
                                         ref[2].astype(np.float32), target, int(L[j]), wl.T, wl.seed, TS)
        assert n[j] <= L[j]
        tally.total += 1
        if (n[j], corr[j]) != (rn, rc):
            assert rm < MARGIN, f"request {j}: ({n[j]}, {corr[j]}) vs ({rn}, {rc}) margin {rm}"
            tally.excluded += 1
    tally.check_fraction()


def test_residual_without_mass_falls_back_to_p():
    # Position 1's target row is the draft's own z = base + W2 W1[anchor], and the draft LSE passed
    # in is 30 nats below the true one: q(x) then exceeds p(x) by a factor e^30 at every id, so the
    # accept test rejects at position 1 and max(0, p - q) has no mass anywhere; the correction is
    # drawn from p instead (the oracle's fallback flag), with the status word left OK.
    wl = W.make_sample_workload("fb", 6, 2, 3000, 16, 1.0, device="cuda", data_seed=17, philox_seed=9,
                                logits_dtype=torch.float32, w_std=0.3)
    t = wl.tensors
    base, W1, W2, anchor, _ = host(wl)
    tok, lse, zat = oracle_drafts(wl)
    def f64(x):  # bf16 bit patterns (uint16) or float32 -> float64
        return ((x.astype(np.uint32) << 16).view(np.float32) if x.dtype == np.uint16 else x).astype(np.float64)

    z1 = f64(base[:, 0]) + f64(W1)[anchor] @ f64(W2).T
    target = np.array(W.np_view(t["target"]), copy=True)
    target[:, 0] = z1.astype(np.float32)
    t["target"].copy_(torch.from_numpy(target).to("cuda"))
    lse_low = (lse - 30.0).astype(np.float32)
    n, corr = verify_both(wl, tok, lse_low, zat)
    assert (n == 0).all()
    for j in range(wl.B):
        _, rc, _, fb = O.verify_request(base, W1, W2, int(anchor[j]), j, tok[j], lse_low[j], zat[j], target, wl.gamma,
                                        wl.T, wl.seed, TS)
        assert fb == 1, j


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_softcap_residuals(T):
    # the draft's capped logits are rebuilt at every rejecting position (the target is taken as given)
    wl = W.make_sample_workload("vcap", 21, 4, 5000, 64, T, device="cuda", data_seed=5, philox_seed=3,
                                target_sigma=0.7, planted=2, w_std=0.3)
    verify_both(wl, *oracle_drafts(wl, softcap=3.0), softcap=3.0)


# ---------------------------------------------------------------- tensor-core residual / bonus draws
# (bf16, rank 64, B >= 64, V % 64 == 0, dense target rows: one CTA per tile walks row blocks of 128
# jobs whose base and target rows are gathered by tensor copies)
@pytest.mark.parametrize("B,gamma,V,T", [(200, 4, 4096, 1.0), (64, 3, 3008, 0.7), (96, 4, 5056, 1.3),
                                         (129, 2, 2048, 0.8)])
def test_tc_jobs(B, gamma, V, T):
    wl = W.make_sample_workload("vtc", B, gamma, V, 64, T, device="cuda", data_seed=B + V, philox_seed=5,
                                target_sigma=0.7, planted=2, w_std=0.3)
    n, corr = verify_both(wl, *oracle_drafts(wl))
    assert (n < gamma).mean() > 0.3  # residual draws were exercised


def test_tc_jobs_verify_len_and_bonus():
    wl = W.make_sample_workload("vtcb", 150, 5, 3008, 64, 1.0, device="cuda", data_seed=23, target_sigma=0.1,
                                gamma_t=6, w_std=0.3)
    tok, lse, zat = oracle_drafts(wl)
    vlen = np.random.default_rng(4).integers(1, 6, wl.B)
    n, corr = verify_both(wl, tok, lse, zat, vlen=vlen)
    assert (n == vlen).sum() > 10 and (corr >= 0).all()  # bonus draws from row L_j + 1


def test_tc_jobs_greedy_bonus():
    wl = W.make_sample_workload("vtcg", 100, 3, 2048, 64, 0.0, device="cuda", data_seed=31, target_sigma=0.01,
                                gamma_t=4, w_std=0.3)
    n, corr = verify_both(wl, *oracle_drafts(wl))
    assert (n == 3).any()


def test_tc_jobs_residual_without_mass_falls_back_to_p():
    # as test_residual_without_mass_falls_back_to_p, on the tensor-core path (bf16, B = 64)
    wl = W.make_sample_workload("vtcfb", 64, 2, 3008, 64, 1.0, device="cuda", data_seed=17, philox_seed=9,
                                w_std=0.3)
    t = wl.tensors
    base, W1, W2, anchor, _ = host(wl)
    tok, lse, zat = oracle_drafts(wl)

    def f64(x):
        return ((x.astype(np.uint32) << 16).view(np.float32) if x.dtype == np.uint16 else x).astype(np.float64)

    z1 = f64(base[:, 0]) + f64(W1)[anchor] @ f64(W2).T
    t["target"][:, 0] = torch.from_numpy(z1.astype(np.float32)).to("cuda").to(torch.bfloat16)
    target = W.np_view(t["target"])
    lse_low = (lse - 30.0).astype(np.float32)
    n, corr = verify_both(wl, tok, lse_low, zat)
    assert (n == 0).all()
    for j in range(0, wl.B, 7):
        _, rc, _, fb = O.verify_request(base, W1, W2, int(anchor[j]), j, tok[j], lse_low[j], zat[j], target, wl.gamma,
                                        wl.T, wl.seed, TS)
        assert fb == 1, j
