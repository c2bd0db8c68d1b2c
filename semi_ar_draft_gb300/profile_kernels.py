"""Launches one kernel of the hot path on its own, for profiler captures (ncu) of a bounded case.

Only the tensors that kernel needs are allocated, so a capture holds a few hundred MB to a few
GB on the device instead of the whole bench step's.  Inputs are the seeded synthetic ones of
workloads.py.  Example (sampler at B = 512, V = 151936, rank 64, 4 steps, three launches):

    python -m semi_ar_draft_gb300.profile_kernels --kernel sample --B 512 --gamma 4 --launches 3

Prints the CUDA-event time of each launch (not valid as a bench number under a profiler).
"""
from __future__ import annotations

import argparse

import torch

from . import api, binding
from . import workloads as W


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=["sample", "verify", "tv", "logits"], required=True)
    ap.add_argument("--B", type=int, default=512)
    ap.add_argument("--gamma", type=int, default=4)
    ap.add_argument("--V", type=int, default=W.VOCAB)
    ap.add_argument("--r", type=int, default=64)
    ap.add_argument("--T", type=float, default=1.0)
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.kernel == "tv":
        wl = W.make_tv_workload(1, args.B, args.gamma, args.V, device=dev)
        t = wl.tensors
        run = lambda: api.accept_rate_tv(t["d"], t["t"], t["keep"])  # noqa: E731
    else:
        wl = W.make_sample_workload("profile", args.B, args.gamma, args.V, args.r, args.T, device=dev,
                                    w_std=0.02)
        t = wl.tensors
        tok, lse, zat, ws = api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], args.T, wl.seed)
        if args.kernel == "sample":
            run = lambda: api.markov_sample_block(t["base"], t["W1"], t["W2"], t["anchor"], args.T, wl.seed)  # noqa: E731
        elif args.kernel == "logits":  # teacher-forced block logits with the drafted tokens as the true ones
            run = lambda: api.markov_block_logits(t["base"], t["W1"], t["W2"], t["anchor"], tok)  # noqa: E731
        else:
            run = lambda: api.verify(t["base"], t["W1"], t["W2"], t["anchor"], tok, lse, zat, t["target"], args.T,  # noqa: E731
                                     wl.seed)
    torch.cuda.synchronize()
    for k in range(args.launches):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        out = run()
        e1.record()
        torch.cuda.synchronize()
        ws = out[-1]
        assert binding.dspark_get_device_status(ws) == 0
        print(f"{args.kernel} launch {k}: {e0.elapsed_time(e1) * 1e3:.1f} us", flush=True)


if __name__ == "__main__":
    main()
