"""Parity of dspark_schedule_verify_len (CUDA) with the oracle: bit-exact L and offsets."""
import numpy as np
import pytest
import torch

import oracle as O
from parity import close
from semi_ar_draft_gb300 import api, binding
from semi_ar_draft_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def check(conf, budget):
    L, off, obj, _ = api.schedule_verify_len(conf, budget)
    rL, roff, robj, _ = O.schedule(conf.cpu().numpy(), budget)
    assert np.array_equal(L.cpu().numpy(), rL)
    assert np.array_equal(off.cpu().numpy(), roff)
    close(obj.cpu().numpy(), [robj], what="objective")


@pytest.mark.parametrize("B,g", [(1, 1), (1, 16), (3, 5), (37, 7), (512, 16), (1024, 16), (2000, 8)])
def test_random_budgets(B, g):
    gen = torch.Generator(device="cuda").manual_seed(B * 31 + g)
    conf = torch.rand((B, g), generator=gen, device="cuda")
    for budget in sorted({B, B + 1, (B * g) // 2, B * g - 1, B * g, B * g + 5}):
        if budget >= B:
            check(conf, budget)


def test_config_b512_budget_2048():
    wl = W.b512_sched(device="cuda", V=1024)  # confidences only
    check(wl.tensors["conf"], 2048)


def test_ties_nan_and_clamp():
    conf = torch.ones((6, 5), device="cuda")
    check(conf, 13)
    conf[1, 2] = float("nan")
    conf[3, 1] = 1.7
    conf[4, 0] = -0.2
    check(conf, 17)
    q = torch.full((40, 8), 0.5, device="cuda")  # many exact ties across rows
    check(q, 100)


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
    for j in range(conf.shape[0]):
        # the oracle on the same float32 values, widened exactly
        r_ell, r_th = O.theta_schedule(conf[j].cpu().numpy().astype(np.float64), prof.cpu().numpy().astype(np.float64))
        assert ell[j] == r_ell, j
        assert np.array_equal(np.isnan(theta[j]), np.isnan(r_th)), j
        ok = ~np.isnan(r_th)
        assert np.array_equal(theta[j][ok], r_th[ok].astype(np.float32)), j  # same IEEE single operations


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
