"""Convenience calls over the binding: allocate outputs and workspace with torch, then call
the C entry point.  Shapes and semantics are those of include/dspark.h."""
from __future__ import annotations

import torch

from . import binding as b


def _wdt(W1):
    return b.F32 if W1 is None else b.dtype_code(W1.dtype)


def make_params(base: torch.Tensor, W1, T: float, seed: int, softcap: float = 0.0) -> b.SampleParams:
    B, gamma, V = base.shape
    r = 0 if W1 is None else W1.shape[1]
    return b.params(B, gamma, V, r, T, seed, b.dtype_code(base.dtype), _wdt(W1), softcap)


def markov_sample_block(base, W1, W2, anchor, T, seed, ws=None, out=None, stream=None, softcap=0.0):
    """Returns (tokens [B,gamma] int32, draft_lse [B,gamma] f32, z_at_tok [B,gamma] f32, workspace)."""
    p = make_params(base, W1, T, seed, softcap)
    B, gamma, _ = base.shape
    dev = base.device
    if out is None:
        out = (torch.empty((B, gamma), dtype=torch.int32, device=dev), torch.empty((B, gamma), device=dev),
               torch.empty((B, gamma), device=dev))
    if ws is None:
        ws = b.workspace(b.dspark_sample_workspace_size(p), dev)
    b.dspark_markov_sample_block(p, base, W1, W2, anchor, out[0], out[1], out[2], ws, stream)
    return out[0], out[1], out[2], ws


def verify(base, W1, W2, anchor, tokens, draft_lse, z_at_tok, target, T, seed, verify_len=None,
           target_row_offsets=None, ws=None, out=None, stream=None, softcap=0.0):
    """Returns (n_accepted [B] int32, correction_token [B] int32, workspace)."""
    p = make_params(base, W1, T, seed, softcap)
    B = base.shape[0]
    gamma_t = 0 if target_row_offsets is not None else target.shape[1]
    dev = base.device
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev))
    if ws is None:
        ws = b.workspace(b.dspark_verify_workspace_size(p, gamma_t), dev)
    b.dspark_verify(p, base, W1, W2, anchor, tokens, draft_lse, z_at_tok, target, gamma_t, verify_len,
                    target_row_offsets, out[0], out[1], ws, stream)
    return out[0], out[1], ws


def markov_sample_block_head(base, W1, W2, anchor, T, seed, kind, hidden, Wg, Wc=None, Wo=None, ws=None,
                             out=None, stream=None, softcap=0.0):
    """Gated / RNN head sampling.  Returns (tokens, draft_lse, z_at_tok, head_vec [B,gamma,r] f32, workspace)."""
    p = make_params(base, W1, T, seed, softcap)
    B, gamma, _ = base.shape
    dev = base.device
    h = b.head(kind, hidden, Wg, Wc, Wo)
    if out is None:
        out = (torch.empty((B, gamma), dtype=torch.int32, device=dev), torch.empty((B, gamma), device=dev),
               torch.empty((B, gamma), device=dev), torch.empty((B, gamma, W1.shape[1]), device=dev))
    if ws is None:
        ws = b.workspace(b.dspark_sample_head_workspace_size(p, h), dev)
    b.dspark_markov_sample_block_head(p, h, base, W1, W2, anchor, out[0], out[1], out[2], out[3], ws, stream)
    return out[0], out[1], out[2], out[3], ws


def verify_head(base, head_vec, W2, anchor, tokens, draft_lse, z_at_tok, target, T, seed, verify_len=None,
                target_row_offsets=None, ws=None, out=None, stream=None, softcap=0.0):
    """dspark_verify for Gated / RNN drafts: q is rebuilt from head_vec [B,gamma,r] f32.
    Returns (n_accepted, correction_token, workspace)."""
    B, gamma, V = base.shape
    r = head_vec.shape[-1]
    p = b.params(B, gamma, V, r, T, seed, b.dtype_code(base.dtype), b.dtype_code(W2.dtype), softcap)
    gamma_t = 0 if target_row_offsets is not None else target.shape[1]
    dev = base.device
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev))
    if ws is None:
        ws = b.workspace(b.dspark_verify_workspace_size(p, gamma_t), dev)
    b.dspark_verify_head(p, base, head_vec, W2, anchor, tokens, draft_lse, z_at_tok, target, gamma_t, verify_len,
                         target_row_offsets, out[0], out[1], ws, stream)
    return out[0], out[1], ws


def accept_rate_tv(d, t, keep, pos_valid=None, want_tau=True, ws=None, out=None, stream=None):
    """d, t [S,A,gamma,V]; keep [S,A] uint8.  Returns (accept_rate, eval_mask, tau or None, workspace)."""
    S, A, gamma, V = d.shape
    dt = b.dtype_code(d.dtype)
    dev = d.device
    if out is None:
        out = (torch.empty((S, A, gamma), device=dev), torch.empty((S, A, gamma), device=dev),
               torch.empty((S, A), device=dev) if want_tau else None)
    if ws is None:
        ws = b.workspace(b.dspark_accept_rate_tv_workspace_size(S, A, gamma, V, dt), dev)
    b.dspark_accept_rate_tv(S, A, gamma, V, dt, d, t, keep, pos_valid, out[0], out[1], out[2], ws, stream)
    return out[0], out[1], out[2], ws


def markov_block_logits(base, W1, W2, anchor, tokens, stream=None, softcap=0.0):
    """Teacher-forced z = base + W2 W1[prev] at every position.  base [B,gamma,V]; returns z [B,gamma,V] f32."""
    p = make_params(base, W1, 1.0, 0, softcap)
    B, gamma, V = base.shape
    z = torch.empty((B, gamma, V), dtype=torch.float32, device=base.device)
    ws = b.workspace(b.dspark_markov_block_logits_workspace_size(p), base.device)
    b.dspark_markov_block_logits(p, base, W1, W2, anchor, tokens, z, ws, stream)
    return z, ws


def tv_l1_loss(accept_rate, eval_mask, decay_gamma=4.0, stream=None):
    """accept_rate, eval_mask [S,A,gamma] f32.  Returns (l1 [S,A,gamma] f32, sums [2] f64: weighted numerator, denominator)."""
    S, A, gamma = accept_rate.shape
    l1 = torch.empty_like(accept_rate)
    sums = torch.empty(2, dtype=torch.float64, device=accept_rate.device)
    b.dspark_tv_l1_loss(S, A, gamma, accept_rate, eval_mask, decay_gamma, l1, sums, stream)
    return l1, sums


def theta_schedule(conf, sps, with_theta=False, stream=None):
    """conf [B,gamma] f32, sps [gamma+1] f32 (device).  Returns (ell [B] int32, theta [B,gamma+1] f32 or None)."""
    B, gamma = conf.shape
    dev = conf.device
    ell = torch.empty(B, dtype=torch.int32, device=dev)
    theta = torch.empty((B, gamma + 1), dtype=torch.float32, device=dev) if with_theta else None
    b.dspark_theta_schedule(B, gamma, conf, sps, ell, theta, stream)
    return ell, theta


def schedule_verify_len(conf, budget, ws=None, out=None, stream=None):
    """conf [B,gamma] f32.  Returns (verify_len [B], offsets [B+1], objective [1], workspace)."""
    B, gamma = conf.shape
    dev = conf.device
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B + 1, dtype=torch.int32, device=dev),
               torch.empty(1, device=dev))
    if ws is None:
        ws = b.workspace(b.dspark_schedule_workspace_size(B, gamma), dev)
    b.dspark_schedule_verify_len(B, gamma, conf, budget, out[0], out[1], out[2], ws, stream)
    return out[0], out[1], out[2], ws
