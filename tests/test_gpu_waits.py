"""Bounded device waits: a grid-wide wait that can never complete gives up after the wait
limit and reports DSPARK_ERR_TIMEOUT in the status word; the context stays usable."""
import pytest
import torch

from semi_ar_draft_gb300 import api, binding
from semi_ar_draft_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    ws = binding.workspace(4096)
    binding.dspark_set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        binding.dspark_selftest_grid_wait(8, 0, ws)
        assert binding.dspark_get_device_status(ws) == 0
        binding.dspark_selftest_grid_wait(8, 1, ws)  # one arrival is missing: nothing completes the wait
        assert binding.dspark_get_device_status(ws) == 4
    finally:
        binding.dspark_set_wait_limit_ns(2_000_000_000)
    wl = W.make_sample_workload("after", 4, 3, 2048, 16, 1.0, device="cuda")
    t = wl.tensors
    tok, _, _, ws2 = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], 1.0, 0)
    assert binding.dspark_get_device_status(ws2) == 0
    assert tok.min().item() >= 0 and tok.max().item() < 2048
