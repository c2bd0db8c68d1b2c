"""Parity of dspark_accept_rate_tv (CUDA) with the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from parity import close
from semi_ar_draft_gb300 import api
from semi_ar_draft_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def check(tv, rows=None):
    t = tv.tensors
    acc, mask, tau, _ = api.accept_rate_tv(t["d"], t["t"], t["keep"], t["pos_valid"])
    torch.cuda.synchronize()
    S, A, g = tv.S, tv.A, tv.gamma
    keep = t["keep"].cpu().numpy()
    pv = None if t["pos_valid"] is None else t["pos_valid"].cpu().numpy()
    g_acc, g_mask, g_tau = acc.cpu().numpy(), mask.cpu().numpy(), tau.cpu().numpy()
    # eval_mask is exact everywhere (integer decisions)
    for s in range(S):
        for a in range(A):
            m, _ = O.eval_mask_tau(np.ones(g), int(keep[s, a]), None if pv is None else pv[s, a])
            assert np.array_equal(g_mask[s, a], m.astype(np.float32))
    blocks = [(s, a) for s in range(S) for a in range(A)] if rows is None else rows
    for s, a in blocks:
        d = W.np_view(t["d"][s, a])
        tt = W.np_view(t["t"][s, a])
        ref = np.array([O.tv_row(d[i], tt[i])[0] for i in range(g)])
        close(g_acc[s, a], ref, what=f"acc[{s},{a}]")
        _, rtau = O.eval_mask_tau(ref, int(keep[s, a]), None if pv is None else pv[s, a])
        close([g_tau[s, a]], [rtau], what=f"tau[{s},{a}]")


@pytest.mark.parametrize("V", [8, 1000, 4096, 33333])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_small(V, dtype):
    check(W.make_tv_workload(2, 5, 3, V, device="cuda", dtype=dtype, data_seed=V, truncate=True, drop=0.3))


def test_vocabulary_beyond_the_copy_ring():
    # 262144 ids: sixteen ring slots per pass, the row far larger than the ring
    check(W.make_tv_workload(1, 2, 2, 262144, device="cuda", data_seed=5))


def test_running_maximum_jumps():
    # Logits far above everything before them (up to 120 against a spread of 3): the running sums are
    # taken against the maximum seen so far, and a group whose terms reach 2^64 restarts them from its
    # own maximum.  Spikes late in a row, early in a row, in d only, in t only, and at the last id.
    tv = W.make_tv_workload(1, 2, 4, 40000, device="cuda", data_seed=11)
    d, t = tv.tensors["d"], tv.tensors["t"]
    d[0, 0, 0, 39000] = 120.0
    t[0, 0, 0, 35000] = 90.0
    d[0, 0, 1, 20000] = 70.0
    t[0, 0, 1, 20001] = 70.0
    d[0, 0, 2, 17000] = 80.0
    t[0, 0, 2, 17000] = 80.0
    d[0, 1, 2, 5] = 100.0
    t[0, 1, 3, :] = -50.0
    t[0, 1, 3, 39999] = 50.0
    check(tv)
    acc = api.accept_rate_tv(d, t, tv.tensors["keep"])[0].cpu().numpy()
    assert acc[0, 0, 2] > 0.99 and acc[0, 0, 0] < 1e-6  # shared spike: p = q; apart: no overlap


def test_identical_rows_give_one():
    tv = W.make_tv_workload(1, 3, 2, 5000, device="cuda")
    t = tv.tensors
    acc, mask, tau, _ = api.accept_rate_tv(t["d"], t["d"].clone(), t["keep"])
    assert torch.allclose(acc, torch.ones_like(acc), atol=2e-6)


def test_full_tv_4x512x8_sampled_rows():
    tv = W.make_tv_workload(device="cuda", truncate=True)
    check(tv, rows=[(0, 0), (1, 77), (2, 300), (3, 511)])


@pytest.mark.parametrize(
    "S,A,g,V",
    [
        (1, 1, 1, 8192),  # one row of one ring slot
        (1, 1, 8, 151936),  # 8 rows: fewer rows than blocks
        (1, 3, 7, 20000),  # partial last slots
        (1, 16, 8, 151936),  # 128 rows
        (1, 32, 8, 151936),  # 256 rows: a ragged second round of rows
        (1, 19, 16, 65536),  # 304 rows: two full rounds
    ],
)
def test_batch_shapes(S, A, g, V):
    check(W.make_tv_workload(S, A, g, V, device="cuda", data_seed=S * 1000 + A * 10 + g, truncate=True, drop=0.2))


def test_repeated_calls_are_bit_identical():
    tv = W.make_tv_workload(1, 16, 8, 151936, device="cuda", data_seed=9)
    t = tv.tensors
    a1 = api.accept_rate_tv(t["d"], t["t"], t["keep"])[0].clone()
    a2 = api.accept_rate_tv(t["d"], t["t"], t["keep"])[0]
    assert torch.equal(a1, a2)


@pytest.mark.parametrize("rho", [0.8, 0.99999])
def test_l1_loss_epilogue(rho):
    # The oracle's side is built from its own accept rates on the raw logits (tv_row) and its own
    # eval mask, never from the CUDA path's outputs.  rho = 0.99999: nearly identical rows, accept
    # rates close to 1, where l1 = 2 (1 - accept) is a small difference of fp32 values.
    tv = W.make_tv_workload(2, 64, 8, 20000, device="cuda", data_seed=3, truncate=True, drop=0.2, rho=rho)
    t = tv.tensors
    S, A, g = tv.S, tv.A, tv.gamma
    acc, mask, _, _ = api.accept_rate_tv(t["d"], t["t"], t["keep"], t["pos_valid"])
    l1, sums = api.tv_l1_loss(acc, mask, 4.0)
    torch.cuda.synchronize()
    keep, pv = t["keep"].cpu().numpy(), t["pos_valid"].cpu().numpy()
    d_all, t_all = W.np_view(t["d"]), W.np_view(t["t"])
    r_acc = np.array([[[O.tv_row(d_all[s_, a, i], t_all[s_, a, i])[0] for i in range(g)] for a in range(A)]
                      for s_ in range(S)])
    r_mask = np.array([[O.eval_mask_tau(r_acc[s_, a], int(keep[s_, a]), pv[s_, a])[0] for a in range(A)]
                       for s_ in range(S)])
    r_l1, r_num, r_den = O.tv_l1_loss(r_acc, r_mask, 4.0)
    # bound from the arithmetic: l1 = 2 (1 - accept) carries twice the accept rate's absolute error,
    # which the TV parity bound holds to 1e-5 accept + 2^-24 (the fp32 spacing near 1)
    bound = 2 * (1e-5 * r_acc + 2.0 ** -24)
    assert (np.abs(l1.cpu().numpy() - r_l1) <= bound).all()
    assert np.array_equal(mask.cpu().numpy(), r_mask.astype(np.float32))
    w = np.exp(-np.arange(g) / 4.0)
    close(sums.cpu().numpy()[1:], [r_den], rtol=1e-12, atol=1e-12, what="weighted mask sum")
    assert abs(float(sums[0]) - r_num) <= float(np.sum(w * r_mask * bound)) + 1e-9
    l1b, sums_b = api.tv_l1_loss(acc, mask, 4.0)
    assert torch.equal(sums, sums_b) and torch.equal(l1, l1b)
