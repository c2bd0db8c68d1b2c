"""Parity of dspark_schedule_verify_len and dspark_theta_schedule (CUDA, fp32) with the fp64
oracle: L, offsets and the chosen prefix are bit-exact except where the oracle's decision margin
is below 1e-5 (counted, under 0.01% of decisions); objective and Theta within 1e-5 relative."""
import numpy as np
import pytest
import torch

import oracle as O
from parity import MARGIN, Tally, close
from semi_ar_draft_gb300 import api, binding
from semi_ar_draft_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def check(conf, budget, tally=None):
    """One call against the oracle.  The selection decisions are the B (gamma - 1) candidate
    positions i >= 2; a survival pair straddling the budget boundary within rounding can be taken
    in the other order (one decision, two requests' L off by one), which is allowed only when the
    oracle's boundary margin is below 1e-5."""
    tally = tally if tally is not None else Tally()
    B, g = conf.shape
    L, off, obj, _ = api.schedule_verify_len(conf, budget)
    rL, roff, robj, mg = O.schedule(conf.cpu().numpy(), budget)
    L, off = L.cpu().numpy(), off.cpu().numpy()
    tally.total += B * max(g - 1, 1)
    if not np.array_equal(L, rL):
        assert mg < MARGIN, (mg, np.nonzero(L != rL))
        tally.excluded += (int(np.abs(L - rL).sum()) + 1) // 2
    # whatever was chosen is a valid selection of the same size
    assert L.min() >= 1 and L.max() <= g and L.sum() == rL.sum()
    assert off[0] == 0 and np.array_equal(np.diff(off), L)
    close(obj.cpu().numpy(), [robj], what="objective")
    return tally


@pytest.mark.parametrize("B,g", [(1, 1), (1, 16), (3, 5), (37, 7), (512, 16), (1024, 16), (2000, 8)])
def test_random_budgets(B, g):
    gen = torch.Generator(device="cuda").manual_seed(B * 31 + g)
    conf = torch.rand((B, g), generator=gen, device="cuda")
    tally = Tally()
    for budget in sorted({B, B + 1, (B * g) // 2, B * g - 1, B * g, B * g + 5}):
        if budget >= B:
            check(conf, budget, tally)
    tally.check_fraction()


def test_config_b512_budget_2048():
    wl = W.b512_sched(device="cuda", V=1024)  # confidences only
    check(wl.tensors["conf"], 2048).check_fraction()


def test_ties_nan_and_clamp():
    # exact ties in both precisions (powers of two, ones): both sides break them by (j, i)
    conf = torch.ones((6, 5), device="cuda")
    check(conf, 13).check_fraction()
    conf[1, 2] = float("nan")
    conf[3, 1] = 1.7
    conf[4, 0] = -0.2
    check(conf, 17).check_fraction()
    q = torch.full((40, 8), 0.5, device="cuda")  # many exact ties across rows
    rL, *_ = O.schedule(q.cpu().numpy(), 100)
    L, *_ = api.schedule_verify_len(q, 100)
    assert np.array_equal(L.cpu().numpy(), rL)


def test_budget_below_b_is_rejected():
    conf = torch.rand((8, 4), device="cuda")
    with pytest.raises(binding.DsparkError) as e:
        api.schedule_verify_len(conf, 7)
    assert e.value.status == 5


# ---------------------------------------------------------------- throughput-aware prefix choice
def _theta_check(c, sps):
    conf = torch.tensor(c, dtype=torch.float32, device="cuda")
    prof = torch.tensor(sps, dtype=torch.float32, device="cuda")
    ell, theta = api.theta_schedule(conf, prof, with_theta=True)
    torch.cuda.synchronize()
    ell, theta = ell.cpu().numpy(), theta.cpu().numpy()
    tally = Tally()
    for j in range(conf.shape[0]):
        # the fp64 oracle on the same float32 values, widened exactly
        r_ell, r_th, mg = O.theta_schedule(conf[j].cpu().numpy().astype(np.float64),
                                           prof.cpu().numpy().astype(np.float64), with_margin=True)
        tally.total += 1
        if ell[j] != r_ell:
            assert mg < MARGIN, (j, ell[j], r_ell, mg)
            tally.excluded += 1
            continue
        assert np.array_equal(np.isnan(theta[j]), np.isnan(r_th)), j
        ok = ~np.isnan(r_th)
        close(theta[j][ok], r_th[ok], atol=0.0, what=f"Theta of request {j}")
    tally.check_fraction()


def test_theta_worked_example_on_gpu():
    # the page's example (c_3 is truncated there; any value keeps the stop at l = 2): choose l = 1
    conf = torch.tensor([[0.8, 0.7, 0.1]], dtype=torch.float32, device="cuda")
    prof = torch.tensor([1.0, 0.95, 0.52, 0.48], dtype=torch.float32, device="cuda")
    ell, theta = api.theta_schedule(conf, prof, with_theta=True)
    assert int(ell[0]) == 1
    assert np.allclose(np.round(theta[0, :3].cpu().numpy(), 2), [1.00, 1.71, 1.23])
    _theta_check(conf.cpu().numpy(), prof.cpu().numpy())


@pytest.mark.parametrize("B,gamma", [(1, 1), (7, 4), (512, 16), (3000, 8)])
def test_theta_matches_oracle(B, gamma):
    rng = np.random.default_rng(B * 100 + gamma)
    c = rng.beta(4.0, 1.5, size=(B, gamma)).astype(np.float32)
    c[rng.random((B, gamma)) < 0.05] = 1.0  # runs of certain tokens
    # a decreasing throughput profile with noise, and a flat stretch (ties between Theta values)
    sps = np.maximum(0.05, 1.0 - 0.06 * np.arange(gamma + 1) + rng.normal(0, 0.02, gamma + 1)).astype(np.float32)
    if gamma >= 4:
        sps[2:4] = sps[2]
    _theta_check(c, sps)
