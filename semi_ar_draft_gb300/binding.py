"""ctypes binding of libdspark (include/dspark.h): argument marshalling only.

Each ``dspark_*`` function here has the C entry point's name and argument order; tensors are
torch CUDA tensors (their device pointers are passed), ``stream`` defaults to torch's current
stream.  A non-OK status raises :class:`DsparkError`.  Every step of the hot path runs in the
CUDA kernels of libdspark; there is no fallback: if the library is not built, loading fails.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from .build import LIB

F32, BF16 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "device wait timed out",
          5: "budget < B", 6: "bad workspace", 7: "token out of range"}


class DsparkError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)} (status {status})")
        self.status = status


HEAD_VANILLA, HEAD_GATED, HEAD_RNN = 0, 1, 2


class Head(C.Structure):
    _fields_ = [("kind", C.c_int), ("d", C.c_int), ("hidden", C.c_void_p), ("Wg", C.c_void_p), ("Wc", C.c_void_p),
                ("Wo", C.c_void_p)]


class SampleParams(C.Structure):
    _fields_ = [("B", C.c_int), ("gamma", C.c_int), ("V", C.c_int), ("r", C.c_int), ("temperature", C.c_float),
                ("seed", C.c_uint64), ("logits_dtype", C.c_int), ("w_dtype", C.c_int), ("softcap", C.c_float)]


_L = None


def lib():
    global _L
    if _L is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"libdspark is not built ({LIB} missing); run __graft_entry__.build()")
        L = C.CDLL(LIB)
        vp, i32, sz, u64 = C.c_void_p, C.c_int, C.c_size_t, C.c_uint64
        P = C.POINTER(SampleParams)
        L.dspark_sample_workspace_size.argtypes = [P]
        L.dspark_sample_workspace_size.restype = sz
        L.dspark_markov_sample_block.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.dspark_markov_sample_block.restype = i32
        L.dspark_markov_sample_block_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
        L.dspark_markov_sample_block_noalloc.restype = i32
        H = C.POINTER(Head)
        L.dspark_sample_head_workspace_size.argtypes = [P, H]
        L.dspark_sample_head_workspace_size.restype = sz
        L.dspark_markov_sample_block_head.argtypes = [P, H, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.dspark_markov_sample_block_head.restype = i32
        L.dspark_verify_head.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp]
        L.dspark_verify_head.restype = i32
        L.dspark_verify_workspace_size.argtypes = [P, i32]
        L.dspark_verify_workspace_size.restype = sz
        L.dspark_verify.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp]
        L.dspark_verify.restype = i32
        L.dspark_accept_rate_tv_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.dspark_accept_rate_tv_workspace_size.restype = sz
        L.dspark_accept_rate_tv.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.dspark_accept_rate_tv.restype = i32
        L.dspark_schedule_workspace_size.argtypes = [i32, i32]
        L.dspark_schedule_workspace_size.restype = sz
        L.dspark_schedule_verify_len.argtypes = [i32, i32, vp, i32, vp, vp, vp, vp, sz, vp]
        L.dspark_schedule_verify_len.restype = i32
        L.dspark_markov_block_logits_workspace_size.argtypes = [C.POINTER(SampleParams)]
        L.dspark_markov_block_logits_workspace_size.restype = sz
        L.dspark_markov_block_logits.argtypes = [C.POINTER(SampleParams), vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.dspark_markov_block_logits.restype = i32
        L.dspark_tv_l1_loss.argtypes = [i32, i32, i32, vp, vp, C.c_float, vp, vp, vp]
        L.dspark_tv_l1_loss.restype = i32
        L.dspark_theta_schedule.argtypes = [i32, i32, vp, vp, vp, vp, vp]
        L.dspark_theta_schedule.restype = i32
        L.dspark_get_device_status.argtypes = [vp, vp, C.POINTER(C.c_int32)]
        L.dspark_get_device_status.restype = i32
        L.dspark_set_wait_limit_ns.argtypes = [u64]
        L.dspark_set_wait_limit_ns.restype = None
        L.dspark_selftest_grid_wait.argtypes = [i32, i32, vp, sz, vp]
        L.dspark_selftest_grid_wait.restype = i32
        L.dspark_status_string.argtypes = [i32]
        L.dspark_status_string.restype = C.c_char_p
        L.dspark_kernel_launches.argtypes = []
        L.dspark_kernel_launches.restype = u64
        _L = L
    return _L


# ------------------------------------------------------------------ marshalling helpers
def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("libdspark takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libdspark takes contiguous tensors")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    raise TypeError(f"libdspark logits/weights are fp32 or bf16, got {dt}")


def _check(st: int, where: str):
    if st != 0:
        raise DsparkError(st, where)


def params(B, gamma, V, r, temperature, seed, logits_dtype, w_dtype, softcap=0.0) -> SampleParams:
    return SampleParams(int(B), int(gamma), int(V), int(r), float(temperature), int(seed) & (2 ** 64 - 1),
                        int(logits_dtype), int(w_dtype), float(softcap))


# ------------------------------------------------------------------ entry points (same names as the C ABI)
def dspark_sample_workspace_size(p: SampleParams) -> int:
    return int(lib().dspark_sample_workspace_size(C.byref(p)))


def dspark_markov_sample_block(p, base_logits, W1, W2, anchor, tokens, draft_lse, draft_logit_at_tok, workspace,
                               stream=None):
    st = lib().dspark_markov_sample_block(C.byref(p), _ptr(base_logits), _ptr(W1), _ptr(W2), _ptr(anchor),
                                          _ptr(tokens), _ptr(draft_lse), _ptr(draft_logit_at_tok), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "dspark_markov_sample_block")


def dspark_markov_sample_block_noalloc(p, base_logits, W1, W2, anchor, tokens, draft_lse, draft_logit_at_tok,
                                       stream=None):
    """Draft sampling with the library's own fixed device scratch (no workspace argument): for
    callers that cannot allocate device memory.  Calls must not overlap on the GPU."""
    st = lib().dspark_markov_sample_block_noalloc(C.byref(p), _ptr(base_logits), _ptr(W1), _ptr(W2), _ptr(anchor),
                                                  _ptr(tokens), _ptr(draft_lse), _ptr(draft_logit_at_tok),
                                                  _stream(stream))
    _check(st, "dspark_markov_sample_block_noalloc")


def head(kind, hidden, Wg, Wc=None, Wo=None) -> Head:
    """A dspark_head over device tensors (kept alive by the caller): hidden [B, gamma, d]."""
    return Head(int(kind), int(hidden.shape[-1]), _ptr(hidden), _ptr(Wg), _ptr(Wc), _ptr(Wo))


def dspark_sample_head_workspace_size(p: SampleParams, h: Head) -> int:
    return int(lib().dspark_sample_head_workspace_size(C.byref(p), C.byref(h)))


def dspark_markov_sample_block_head(p, h, base_logits, W1, W2, anchor, tokens, draft_lse, draft_logit_at_tok,
                                    head_vec, workspace, stream=None):
    st = lib().dspark_markov_sample_block_head(C.byref(p), C.byref(h), _ptr(base_logits), _ptr(W1), _ptr(W2),
                                               _ptr(anchor), _ptr(tokens), _ptr(draft_lse), _ptr(draft_logit_at_tok),
                                               _ptr(head_vec), _ptr(workspace),
                                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "dspark_markov_sample_block_head")


def dspark_verify_head(p, base_logits, head_vec, W2, anchor, tokens, draft_lse, draft_logit_at_tok, target_logits,
                       gamma_t, verify_len, target_row_offsets, n_accepted, correction_token, workspace, stream=None):
    st = lib().dspark_verify_head(C.byref(p), _ptr(base_logits), _ptr(head_vec), _ptr(W2), _ptr(anchor),
                                  _ptr(tokens), _ptr(draft_lse), _ptr(draft_logit_at_tok), _ptr(target_logits),
                                  int(gamma_t), _ptr(verify_len), _ptr(target_row_offsets), _ptr(n_accepted),
                                  _ptr(correction_token), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "dspark_verify_head")


def dspark_verify_workspace_size(p: SampleParams, gamma_t: int) -> int:
    return int(lib().dspark_verify_workspace_size(C.byref(p), int(gamma_t)))


def dspark_verify(p, base_logits, W1, W2, anchor, tokens, draft_lse, draft_logit_at_tok, target_logits, gamma_t,
                  verify_len, target_row_offsets, n_accepted, correction_token, workspace, stream=None):
    st = lib().dspark_verify(C.byref(p), _ptr(base_logits), _ptr(W1), _ptr(W2), _ptr(anchor), _ptr(tokens),
                             _ptr(draft_lse), _ptr(draft_logit_at_tok), _ptr(target_logits), int(gamma_t),
                             _ptr(verify_len), _ptr(target_row_offsets), _ptr(n_accepted), _ptr(correction_token),
                             _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "dspark_verify")


def dspark_accept_rate_tv_workspace_size(S, A, gamma, V, dtype) -> int:
    return int(lib().dspark_accept_rate_tv_workspace_size(S, A, gamma, V, dtype))


def dspark_accept_rate_tv(S, A, gamma, V, dtype, draft_logits, target_logits, block_keep, pos_valid, accept_rate,
                          eval_mask, tau, workspace, stream=None):
    st = lib().dspark_accept_rate_tv(int(S), int(A), int(gamma), int(V), int(dtype), _ptr(draft_logits),
                                     _ptr(target_logits), _ptr(block_keep), _ptr(pos_valid), _ptr(accept_rate),
                                     _ptr(eval_mask), _ptr(tau), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "dspark_accept_rate_tv")


def dspark_schedule_workspace_size(B, gamma) -> int:
    return int(lib().dspark_schedule_workspace_size(int(B), int(gamma)))


def dspark_schedule_verify_len(B, gamma, conf, budget, verify_len, offsets, objective, workspace, stream=None):
    st = lib().dspark_schedule_verify_len(int(B), int(gamma), _ptr(conf), int(budget), _ptr(verify_len),
                                          _ptr(offsets), _ptr(objective), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "dspark_schedule_verify_len")


def dspark_markov_block_logits_workspace_size(p) -> int:
    return int(lib().dspark_markov_block_logits_workspace_size(C.byref(p)))


def dspark_markov_block_logits(p, base, W1, W2, anchor, tokens, z_out, workspace, stream=None):
    st = lib().dspark_markov_block_logits(C.byref(p), _ptr(base), _ptr(W1), _ptr(W2), _ptr(anchor), _ptr(tokens),
                                          _ptr(z_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(stream))
    _check(st, "dspark_markov_block_logits")


def dspark_tv_l1_loss(S, A, gamma, accept_rate, eval_mask, decay_gamma, l1, sums, stream=None):
    st = lib().dspark_tv_l1_loss(int(S), int(A), int(gamma), _ptr(accept_rate), _ptr(eval_mask), float(decay_gamma),
                                 _ptr(l1), _ptr(sums), _stream(stream))
    _check(st, "dspark_tv_l1_loss")


def dspark_theta_schedule(B, gamma, conf, sps, ell, theta=None, stream=None):
    st = lib().dspark_theta_schedule(int(B), int(gamma), _ptr(conf), _ptr(sps), _ptr(ell), _ptr(theta),
                                     _stream(stream))
    _check(st, "dspark_theta_schedule")


def dspark_get_device_status(workspace, stream=None) -> int:
    out = C.c_int32(0)
    st = lib().dspark_get_device_status(_ptr(workspace), _stream(stream), C.byref(out))
    _check(st, "dspark_get_device_status")
    return int(out.value)


def dspark_set_wait_limit_ns(ns: int):
    lib().dspark_set_wait_limit_ns(int(ns))


def dspark_selftest_grid_wait(nblocks, missing, workspace, stream=None):
    st = lib().dspark_selftest_grid_wait(int(nblocks), int(missing), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "dspark_selftest_grid_wait")


def dspark_kernel_launches() -> int:
    return int(lib().dspark_kernel_launches())


def dspark_status_string(s: int) -> str:
    return lib().dspark_status_string(int(s)).decode()


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A caller-owned workspace (256-byte aligned: torch's CUDA allocator aligns to 512)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
