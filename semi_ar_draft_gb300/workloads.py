"""Seeded synthetic inputs for the DSpark hot path.

This module holds no arithmetic of the method: it only draws random tensors with
the shapes, dtypes and value distributions of the workloads below and hands the
same bytes to the CUDA library and to the CPU oracle.  It is the only code the
two sides share.  Generation uses ``torch.Generator`` on the requested device;
full-size tensors are drawn on the GPU in slices so the host never holds them.

Workloads (all synthetic; the pages run trained models that are not available):
  tiny        B=1, gamma=4, V=1024, r=16, fp32 base ~N(0,2), W ~N(0,0.02),
              target = base + N(0,1), T in {0, 1}
  b32_r64     B=32, gamma=8, V=151936, r=64, bf16 base ~N(0,3) with 5 planted
              peaks (+8) per position, W ~N(0,0.02), T=1, target = base + N(0,1)
  b128_r256   B=128, gamma=16, V=151936, r=256, bf16 base ~N(0,3), T=0.7,
              target = base + N(0, sigma_i), sigma_i = 0.5 + 2.5 (i-1)/15
  tv_4x512x8  S=4, A=512, gamma=8, V=151936, d = 3x, t = 3(0.8x + 0.6y), x,y iid
              N(0,1) in bf16 (correlation 0.8), 10% of anchors with keep=0
  b512_sched  B=512, gamma=16, V=151936, r=64, T=1, bf16 base ~N(0,3), target =
              base + N(0,1), confidences Beta(8,2) x 0.93^(i-1), budget 2048
  heads       (make_head_inputs) hidden states [B, gamma, d] ~N(0,1) and Gated / RNN head
              weights ~N(0, w_std) in the sampler's weight dtype
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

VOCAB = 151936


@dataclass
class SampleWorkload:
    name: str
    B: int
    gamma: int
    V: int
    r: int
    T: float
    seed: int  # the Philox key of the method's own random draws
    logits_dtype: torch.dtype
    w_dtype: torch.dtype
    gamma_t: int
    budget: int | None = None
    tensors: dict = field(default_factory=dict)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device, dtype=torch.float32):
    return torch.randn(shape, generator=g, device=device, dtype=dtype) * std


def make_sample_workload(name: str, B: int, gamma: int, V: int, r: int, T: float, *, device="cpu",
                         data_seed: int = 0, philox_seed: int = 0, logits_dtype=torch.bfloat16,
                         w_dtype=torch.bfloat16, base_std: float = 3.0, planted: int = 0,
                         planted_height: float = 8.0, target_sigma=1.0, gamma_t: int | None = None,
                         conf: bool = False, budget: int | None = None, w_std: float = 0.02) -> SampleWorkload:
    """Draws base logits [B,gamma,V], W1/W2 [V,r], anchors [B], target logits
    [B,gamma_t,V] (target = base + noise; noise std per position is
    ``target_sigma(i)`` when callable), and optionally confidences [B,gamma]."""
    gamma_t = gamma if gamma_t is None else gamma_t
    g = _gen(device, data_seed)
    base = torch.empty((B, gamma, V), dtype=logits_dtype, device=device)
    target = torch.empty((B, gamma_t, V), dtype=logits_dtype, device=device)
    for j in range(B):
        blk = _normal((gamma, V), base_std, g, device)
        if planted:
            keys = torch.rand((gamma, V), generator=g, device=device)
            idx = keys.topk(planted, dim=1).indices
            blk.scatter_add_(1, idx, torch.full(idx.shape, planted_height, device=device))
        base[j] = blk.to(logits_dtype)
        b32 = base[j].float()
        for i in range(gamma_t):
            src = b32[min(i, gamma - 1)]
            sig = target_sigma(i + 1) if callable(target_sigma) else float(target_sigma)
            target[j, i] = (src + _normal((V,), sig, g, device)).to(logits_dtype)
    if r > 0:
        W1 = _normal((V, r), w_std, g, device).to(w_dtype)
        W2 = _normal((V, r), w_std, g, device).to(w_dtype)
    else:
        W1 = W2 = None
    anchor = torch.randint(0, V, (B,), generator=g, device=device, dtype=torch.int32)
    t = {"base": base, "W1": W1, "W2": W2, "anchor": anchor, "target": target}
    if conf:
        # Beta(8,2) = G8 / (G8 + G2), G_k = sum of k unit exponentials.
        u = torch.rand((B, gamma, 10), generator=g, device=device, dtype=torch.float64)
        e = -torch.log(u)
        g8, g2 = e[..., :8].sum(-1), e[..., 8:].sum(-1)
        decay = torch.tensor([0.93 ** i for i in range(gamma)], dtype=torch.float64, device=device)
        t["conf"] = (g8 / (g8 + g2) * decay).to(torch.float32).contiguous()
    return SampleWorkload(name, B, gamma, V, r, T, philox_seed, logits_dtype, w_dtype, gamma_t, budget, t)


def sigma_linear(i: int, gamma: int = 16) -> float:
    """Target noise grows linearly from 0.5 at position 1 to 3.0 at position gamma."""
    return 0.5 + 2.5 * (i - 1) / max(gamma - 1, 1)


def tiny(T: float, device="cpu", data_seed=0) -> SampleWorkload:
    return make_sample_workload("tiny", 1, 4, 1024, 16, T, device=device, data_seed=data_seed,
                                logits_dtype=torch.float32, w_dtype=torch.float32, base_std=2.0)


def b32_r64(device="cpu", data_seed=0, V=VOCAB, B=32) -> SampleWorkload:
    return make_sample_workload("b32_r64", B, 8, V, 64, 1.0, device=device, data_seed=data_seed, planted=5,
                                conf=True, budget=B * 8)


def b128_r256(device="cpu", data_seed=0, V=VOCAB, B=128) -> SampleWorkload:
    return make_sample_workload("b128_r256", B, 16, V, 256, 0.7, device=device, data_seed=data_seed,
                                target_sigma=lambda i: sigma_linear(i, 16), conf=True, budget=B * 16)


def b512_sched(device="cpu", data_seed=0, V=VOCAB, B=512, budget=2048) -> SampleWorkload:
    return make_sample_workload("b512_sched", B, 16, V, 64, 1.0, device=device, data_seed=data_seed,
                                conf=True, budget=budget)


HEAD_GATED, HEAD_RNN = 1, 2


def make_head_inputs(wl: SampleWorkload, kind: int, d: int, *, data_seed: int = 0, w_std: float = 0.2,
                     h_std: float = 1.0, device=None) -> dict:
    """Hidden states [B, gamma, d] and the head's weights for workload ``wl`` (its r and
    weight dtype): gated Wg [r, d + r]; rnn Wg, Wc, Wo [r, 2r + d]."""
    device = device if device is not None else wl.tensors["base"].device
    g = _gen(device, 7919 + data_seed)
    r = wl.r
    cols = d + r if kind == HEAD_GATED else 2 * r + d
    out = {"hidden": _normal((wl.B, wl.gamma, d), h_std, g, device).to(wl.w_dtype)}
    names = ["Wg"] if kind == HEAD_GATED else ["Wg", "Wc", "Wo"]
    for n in names:
        out[n] = _normal((r, cols), w_std, g, device).to(wl.w_dtype)
    return out


@dataclass
class TVWorkload:
    name: str
    S: int
    A: int
    gamma: int
    V: int
    dtype: torch.dtype
    tensors: dict = field(default_factory=dict)


def make_tv_workload(S=4, A=512, gamma=8, V=VOCAB, *, device="cpu", data_seed=0, dtype=torch.bfloat16,
                     rho=0.8, scale=3.0, drop=0.1, truncate=False) -> TVWorkload:
    """d = scale*x, t = scale*(rho x + sqrt(1-rho^2) y); keep = 0 for a `drop`
    fraction of (s,a); with `truncate`, pos_valid[s,a,:] is 1 up to a random
    point per block and 0 after it (exercises the cumprod)."""
    g = _gen(device, data_seed)
    d = torch.empty((S, A, gamma, V), dtype=dtype, device=device)
    t = torch.empty((S, A, gamma, V), dtype=dtype, device=device)
    c = math.sqrt(1.0 - rho * rho)
    for s in range(S):
        for a0 in range(0, A, 64):
            a1 = min(A, a0 + 64)
            x = torch.randn((a1 - a0, gamma, V), generator=g, device=device)
            y = torch.randn((a1 - a0, gamma, V), generator=g, device=device)
            d[s, a0:a1] = (scale * x).to(dtype)
            t[s, a0:a1] = (scale * (rho * x + c * y)).to(dtype)
    keep = (torch.rand((S, A), generator=g, device=device) >= drop).to(torch.uint8)
    pos_valid = None
    if truncate:
        cut = torch.randint(1, gamma + 2, (S, A, 1), generator=g, device=device)
        pos_valid = (torch.arange(gamma, device=device).view(1, 1, gamma) < cut).to(torch.uint8).contiguous()
    return TVWorkload("tv_4x512x8", S, A, gamma, V, dtype, {"d": d, "t": t, "keep": keep, "pos_valid": pos_valid})


# ------------------------------------------------------------------ host views
def np_view(x: torch.Tensor):
    """Host numpy view of a tensor for the oracle: bf16 as uint16 bit patterns."""
    import numpy as np

    x = x.detach().contiguous().cpu()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy()
