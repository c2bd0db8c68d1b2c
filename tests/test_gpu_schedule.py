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
