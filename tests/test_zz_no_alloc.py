"""The no-allocation sampling entry point (dspark_markov_sample_block_noalloc) gives the same
drafts as the workspace entry point, on two calls in a row that share its fixed scratch.

It exists for callers that cannot allocate device memory themselves (for instance a plug-in
whose process owns all device memory through its own pool), so it takes no workspace; the
library keeps a fixed scratch array in device memory instead.  This file is collected last."""
import numpy as np
import pytest
import torch

from parity import close
from semi_ar_draft_gb300 import api, binding
from semi_ar_draft_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(wl):
    B, g = wl.B, wl.gamma
    return (torch.full((B, g), -7, dtype=torch.int32, device="cuda"), torch.full((B, g), 7.0, device="cuda"),
            torch.full((B, g), 7.0, device="cuda"))


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_noalloc_matches_workspace_entry_point_twice(T):
    wl = W.make_sample_workload("noalloc", 37, 4, 6000, 64, T, device="cuda", data_seed=21, philox_seed=5, planted=2)
    t = wl.tensors
    ref_tok, ref_lse, ref_zat, _ = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], T, wl.seed)
    ref_tok, ref_lse, ref_zat = ref_tok.cpu().numpy(), ref_lse.cpu().numpy(), ref_zat.cpu().numpy()
    p = api.make_params(t["base"], t["W1"], T, wl.seed)
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        tok, lse, zat = _outputs(wl)
        binding.dspark_markov_sample_block_noalloc(p, t["base"], t["W1"], t["W2"], t["anchor"], tok, lse, zat)
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), ref_tok)
        if T > 0:
            close(lse.cpu().numpy(), ref_lse, what="draft_lse")
        else:
            assert np.isnan(lse.cpu().numpy()).all()
        close(zat.cpu().numpy(), ref_zat, what="z_at_tok")


def test_noalloc_rejects_oversized_scratch():
    # B = 4096 requests over V = 151936 need more scratch than the fixed array holds
    p = binding.params(4096, 2, 151936, 0, 1.0, 0, binding.BF16, binding.BF16)
    assert binding.dspark_sample_workspace_size(p) > (8 << 20)
    dummy = torch.zeros(16, device="cuda")
    with pytest.raises(binding.DsparkError) as e:
        binding.dspark_markov_sample_block_noalloc(p, dummy, None, None, dummy, dummy, dummy, dummy)
    assert e.value.status == 2
