"""The C-ABI library loads and exports every entry point that include/dspark.h declares, and
the host-side argument checks answer without touching a GPU."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


@pytest.fixture(scope="module")
def L():
    from semi_ar_draft_gb300 import build

    build.build()
    from semi_ar_draft_gb300 import binding

    return binding.lib()


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared()
    for n in ["dspark_markov_sample_block", "dspark_verify", "dspark_accept_rate_tv", "dspark_schedule_verify_len"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared():
        assert hasattr(L, n), n


def test_status_strings(L):
    from semi_ar_draft_gb300 import binding as b

    assert b.dspark_status_string(0) == "ok"
    assert "budget" in b.dspark_status_string(5)


def test_workspace_sizes(L):
    from semi_ar_draft_gb300 import binding as b

    p = b.params(32, 8, 151936, 64, 1.0, 0, b.BF16, b.BF16)
    nt = (151936 + 1023) // 1024
    assert b.dspark_sample_workspace_size(p) >= 256 + 32 * 4 + 32 * nt * 16
    assert b.dspark_verify_workspace_size(p, 8) >= 256 + 32 * nt * 16
    assert b.dspark_sample_workspace_size(b.params(0, 8, 10, 0, 1.0, 0, 0, 0)) == 0  # invalid -> 0
    assert b.dspark_schedule_workspace_size(512, 16) >= 256


def test_host_validation_needs_no_gpu(L):
    from semi_ar_draft_gb300 import binding as b

    vp = C.c_void_p
    fake = vp(0x1000)
    bad = b.params(0, 8, 100, 0, 1.0, 0, 0, 0)
    assert L.dspark_markov_sample_block(C.byref(bad), fake, None, None, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    neg_t = b.params(4, 8, 100, 0, -1.0, 0, 0, 0)
    assert L.dspark_markov_sample_block(C.byref(neg_t), fake, None, None, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    big = b.params(5000, 8, 100, 0, 1.0, 0, 0, 0)
    assert L.dspark_markov_sample_block(C.byref(big), fake, None, None, fake, fake, fake, fake, fake, 1 << 20, None) == 2
    ok = b.params(4, 8, 100, 8, 1.0, 0, 0, 0)
    # r > 0 without weights
    assert L.dspark_markov_sample_block(C.byref(ok), fake, None, None, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    # workspace too small / misaligned
    assert L.dspark_markov_sample_block(C.byref(ok), fake, fake, fake, fake, fake, fake, fake, fake, 16, None) == 6
    assert L.dspark_markov_sample_block(C.byref(ok), fake, fake, fake, fake, fake, fake, fake, vp(0x1001), 1 << 20, None) == 6
    # scheduler: budget < B, too many cells
    assert L.dspark_schedule_verify_len(8, 4, fake, 7, fake, fake, None, fake, 1 << 20, None) == 5
    assert L.dspark_theta_schedule(0, 4, fake, fake, fake, None, None) == 1  # B < 1
    assert L.dspark_theta_schedule(8, 4, fake, None, fake, None, None) == 1  # no SPS profile
    assert L.dspark_schedule_verify_len(4096, 8, fake, 8192, fake, fake, None, fake, 1 << 20, None) == 2
    # TV: bad dtype
    assert L.dspark_accept_rate_tv(1, 1, 1, 8, 7, fake, fake, fake, None, fake, fake, None, fake, 1 << 20, None) == 1
    # L1 term: no sums buffer, decay not positive
    assert L.dspark_tv_l1_loss(1, 4, 8, fake, fake, C.c_float(4.0), None, None, None) == 1
    assert L.dspark_tv_l1_loss(1, 4, 8, fake, fake, C.c_float(0.0), None, fake, None) == 1
    # teacher-forced block logits: bad params, r > 0 without weights, tokens missing, workspace
    assert L.dspark_markov_block_logits(C.byref(bad), fake, None, None, fake, fake, fake, fake, 1 << 20, None) == 1
    assert L.dspark_markov_block_logits(C.byref(ok), fake, None, None, fake, fake, fake, fake, 1 << 20, None) == 1
    assert L.dspark_markov_block_logits(C.byref(ok), fake, fake, fake, fake, None, fake, fake, 1 << 20, None) == 1
    assert L.dspark_markov_block_logits(C.byref(ok), fake, fake, fake, fake, fake, fake, fake, 16, None) == 6
    assert b.dspark_markov_block_logits_workspace_size(ok) >= 256
    assert b.dspark_markov_block_logits_workspace_size(bad) == 0
    # verify: dense layout needs gamma_t >= 1
    assert L.dspark_verify(C.byref(ok), fake, fake, fake, fake, fake, fake, fake, fake, 0, None, None, fake, fake,
                           fake, 1 << 20, None) == 1


def test_head_host_validation_needs_no_gpu(L):
    from semi_ar_draft_gb300 import binding as b

    vp = C.c_void_p
    fake = vp(0x1000)
    ok = b.params(4, 8, 100, 8, 1.0, 0, 0, 0)
    gated = b.Head(b.HEAD_GATED, 16, 0x1000, 0x1000, None, None)
    rnn = b.Head(b.HEAD_RNN, 16, 0x1000, 0x1000, 0x1000, 0x1000)
    size_g = b.dspark_sample_head_workspace_size(ok, gated)
    size_r = b.dspark_sample_head_workspace_size(ok, rnn)
    # the head adds the hidden-state pre-activations: 4 x 8 x (1 or 3) x 8 floats
    assert size_g >= b.dspark_sample_workspace_size(ok) + 4 * 8 * 8 * 4
    assert size_r >= b.dspark_sample_workspace_size(ok) + 3 * 4 * 8 * 8 * 4
    for bad in [b.Head(7, 16, 0x1000, 0x1000, None, None),        # unknown kind
                b.Head(b.HEAD_GATED, 0, 0x1000, 0x1000, None, None),  # d < 1
                b.Head(b.HEAD_GATED, 16, None, 0x1000, None, None),    # no hidden state
                b.Head(b.HEAD_RNN, 16, 0x1000, 0x1000, None, 0x1000)]:  # rnn without Wc
        assert b.dspark_sample_head_workspace_size(ok, bad) == 0
        assert L.dspark_markov_sample_block_head(C.byref(ok), C.byref(bad), fake, fake, fake, fake, fake, fake, fake,
                                                 None, fake, 1 << 20, None) == 1
    r0 = b.params(4, 8, 100, 0, 1.0, 0, 0, 0)  # a head needs r >= 1
    assert L.dspark_markov_sample_block_head(C.byref(r0), C.byref(gated), fake, fake, fake, fake, fake, fake, fake,
                                             None, fake, 1 << 20, None) == 1
    # workspace one byte short of the head's size
    assert L.dspark_markov_sample_block_head(C.byref(ok), C.byref(rnn), fake, fake, fake, fake, fake, fake, fake,
                                             None, fake, size_r - 1, None) == 6
    # verify_head: head vectors required
    assert L.dspark_verify_head(C.byref(ok), fake, None, fake, fake, fake, fake, fake, fake, 8, None, None, fake, fake,
                                fake, 1 << 20, None) == 1


def test_kernel_launch_counter(L):
    from semi_ar_draft_gb300 import binding as b

    # readable without a GPU; host-validation failures enqueue nothing and do not count
    n0 = b.dspark_kernel_launches()
    bad = b.params(0, 8, 100, 0, 1.0, 0, 0, 0)
    fake = C.c_void_p(0x1000)
    assert L.dspark_markov_sample_block(C.byref(bad), fake, None, None, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    assert b.dspark_kernel_launches() == n0 >= 0


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import importlib

    from semi_ar_draft_gb300 import binding

    monkeypatch.setattr(binding, "LIB", str(tmp_path / "nope.so"))
    monkeypatch.setattr(binding, "_L", None)
    with pytest.raises(RuntimeError):
        binding.lib()
    importlib.reload(binding)
