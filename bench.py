"""Benchmark of the DSpark hot path on one or more GPUs (one process per GPU).

A step is one pass of the whole hot path over one batch of the b512_sched workload (B=512
requests, gamma=16, V=151936, Markov rank 64, bf16 logits and weights, T=1, a verify budget of
2048 tokens), the largest configuration that fits one GPU:
  schedule  (dspark_schedule_verify_len: verify lengths L_j under the budget)
  sample    (dspark_markov_sample_block)
  verify    (dspark_verify of the scheduled prefixes)
  tv        (dspark_accept_rate_tv on the batch's draft/target logits, eval_mask and tau)
metric = drafted tokens per second = N * B * gamma / step time (replicas: every rank runs its own
batch, "weak" scaling); verified tokens per second (sum L_j over schedule + verify) is reported
beside it.  Inputs are synthetic, seeded, resident in HBM before timing; L2 is flushed (256 MB
write) before every step, outside the per-step CUDA-event interval.

Other workloads of the same path can be timed with --workload (b32_r64: B=32, gamma=8, every
position verified; b128_r256: B=128, gamma=16, rank 256, T=0.7).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft tokens/s (sample+verify) at V=151936; achieved HBM GB/s vs peak"
WORKLOAD = "b512_sched"
WORKLOADS = ("b32_r64", "b128_r256", "b512_sched")
E2E_STEPS = 30  # steps per end-to-end window (each step copies the batch's inputs in: 5 GB at b512_sched)
KERNEL_SOURCES = {
    "sample": ["sample.cu", "sample_tc.cu", "tc05.cuh", "markov_tile.cuh", "common.cuh"],
    "verify": ["verify.cu", "sample_tc.cu", "tc05.cuh", "markov_tile.cuh", "common.cuh"],
    "tv": ["tv.cu", "common.cuh"],
    "schedule": ["schedule.cu", "common.cuh"],
}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _code_only(text: str) -> str:
    """The source without comments or blank lines, each line's whitespace collapsed: a comment or
    layout edit keeps the hash."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip())


def source_hash(kernel: str) -> str:
    """Hash of the code (not the comments) of a kernel's sources: profiled traffic applies while it holds."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "semi_ar_draft_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(kernel)
    except Exception:
        return None
    if not rec or rec.get("source_hash") != source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def wait_first(self, timeout_s: float = 5.0):
        """Block until nvidia-smi has printed its first sample (so the timed window is covered)."""
        t_end = time.perf_counter() + timeout_s
        while self.proc and not self.lines and time.perf_counter() < t_end:
            time.sleep(0.02)

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        """Median SM clock and throttle reasons over the samples taken inside [t0, t1]."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if not (t0 <= ts <= t1):
                continue
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_bytes(wl, n_rejected: int, n_verified: int):
    """Bytes each call must move (bf16): sample reads every base row and W2 once; verify reads the
    n_verified scheduled target rows, plus a base and a target row per rejection (and W2 once)."""
    B, g, V, r = wl.B, wl.gamma, wl.V, wl.r
    e = 2  # bf16
    sample = B * g * V * e + V * r * e + B * g * r * e + B * g * 12
    verify = n_verified * V * e + n_rejected * V * (e + e) + (V * r * e if n_rejected else 0) + B * 8
    tv = 2 * B * g * V * e + B * g * 8 + B * 4
    schedule = B * g * 4 + (2 * B + 1) * 4
    return {"sample": sample, "verify": verify, "tv": tv, "schedule": schedule}


def run_cpu_baseline(wl_host, seconds: float = 15.0, wl_name: str = WORKLOAD, T: float = 1.0, budget=None):
    """The oracle, as it stands, on a bounded sample of the same batch: the scheduler over the
    batch (the workload's budget), then whole requests of the step (sample, verify of the
    scheduled prefix, their accept-rate rows)."""
    import numpy as np

    import oracle as O

    base, W1, W2, anchor, target, conf = wl_host
    B, g, V = base.shape
    t0 = time.perf_counter()
    L, _, _, _ = O.schedule(conf, budget if budget else B * g)
    done = 0
    for j in range(B):
        tok, lse, zat, _ = O.sample_request(base, W1, W2, int(anchor[j]), j, T, 0, 1024)
        O.verify_request(base, W1, W2, int(anchor[j]), j, tok, lse.astype(np.float32), zat.astype(np.float32), target,
                         int(L[j]), T, 0, 1024)
        for i in range(g):
            O.tv_row(base[j, i], target[j, i])
        done += 1
        if time.perf_counter() - t0 > seconds:
            break
    el = time.perf_counter() - t0
    return {"value": done * g / el, "unit": "draft tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of {B} requests of {wl_name} (sample+verify+tv rows) + schedule over the batch, "
                      f"single-threaded C oracle, {el:.1f} s"}


def host_workload(device, data_seed=0, name=WORKLOAD):
    from semi_ar_draft_gb300 import workloads as W

    wl = getattr(W, name)(device=device, data_seed=data_seed)
    t = wl.tensors
    return wl, (W.np_view(t["base"]), W.np_view(t["W1"]), W.np_view(t["W2"]), t["anchor"].cpu().numpy(),
                W.np_view(t["target"]), t["conf"].cpu().numpy())


def reference_arm(args, rank, world):
    if rank != 0:
        return
    import numpy as np  # noqa: F401

    wl, host = host_workload("cpu", name=args.workload)
    B, g = wl.B, wl.gamma
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state
    # each step is a bounded sample (whole requests) of the batch; the run stops after ~2 minutes
    budget_s = 120.0
    per_step = min(5.0, budget_s / max(args.steps, 1))
    vals = []
    samples = []
    t_start = time.perf_counter()
    for _ in range(args.steps):
        cb = run_cpu_baseline(host, seconds=per_step, wl_name=args.workload, T=wl.T, budget=wl.budget)
        vals.append(cb["value"])
        samples.append(cb["sample"])
        if time.perf_counter() - t_start > budget_s and len(vals) >= 3:
            break
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "draft tokens/s", "n_gpus": args.gpus,
            "steps": len(vals), "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": B * g / v * 1e3,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "gamma": g, "V": wl.V, "r": wl.r, "T": wl.T},
            "cpu_baseline": {"value": v, "unit": "draft tokens/s", "cores": 1, "kind": "oracle", "sample": samples[0]},
            "e2e": {"value": v, "unit": "draft tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD, choices=WORKLOADS)
    args = ap.parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import torch

    from semi_ar_draft_gb300 import api, binding, shard
    from semi_ar_draft_gb300 import build as B_

    B_.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    # weak scaling: rank k runs its own shard (requests k*B .. k*B+B-1 of the job's batch):
    # its own seeded inputs and its own Philox key; no collective touches the data path
    wl, host = host_workload(dev, data_seed=rank, name=args.workload)
    t = wl.tensors
    B, g, V = wl.B, wl.gamma, wl.V
    budget = wl.budget if wl.budget else B * g
    base, W1, W2, anchor, target, conf = t["base"], t["W1"], t["W2"], t["anchor"], t["target"], t["conf"]
    d4 = base.view(1, B, g, V)
    t4 = target.view(1, B, g, V)
    keep = torch.ones((1, B), dtype=torch.uint8, device=dev)
    # outputs and workspaces allocated once (caller-owned)
    Lout = torch.empty(B, dtype=torch.int32, device=dev)
    off = torch.empty(B + 1, dtype=torch.int32, device=dev)
    obj = torch.empty(1, device=dev)
    tok = torch.empty((B, g), dtype=torch.int32, device=dev)
    lse = torch.empty((B, g), device=dev)
    zat = torch.empty((B, g), device=dev)
    nacc = torch.empty(B, dtype=torch.int32, device=dev)
    corr = torch.empty(B, dtype=torch.int32, device=dev)
    acc = torch.empty((1, B, g), device=dev)
    emask = torch.empty((1, B, g), device=dev)
    tau = torch.empty((1, B), device=dev)
    p = api.make_params(base, W1, wl.T, shard.rank_seed(wl.seed, rank))
    ws_s = binding.workspace(binding.dspark_schedule_workspace_size(B, g), dev)
    ws_a = binding.workspace(binding.dspark_sample_workspace_size(p), dev)
    ws_v = binding.workspace(binding.dspark_verify_workspace_size(p, g), dev)
    ws_t = binding.workspace(binding.dspark_accept_rate_tv_workspace_size(1, B, g, V, binding.BF16), dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step(src=None):
        bs, ts, cs, an = (base, target, conf, anchor) if src is None else src
        d_, t_ = bs.view(1, B, g, V), ts.view(1, B, g, V)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        ev[0].record()
        binding.dspark_schedule_verify_len(B, g, cs, budget, Lout, off, obj, ws_s)
        ev[1].record()
        binding.dspark_markov_sample_block(p, bs, W1, W2, an, tok, lse, zat, ws_a)
        ev[2].record()
        binding.dspark_verify(p, bs, W1, W2, an, tok, lse, zat, ts, g, Lout, None, nacc, corr, ws_v)
        ev[3].record()
        binding.dspark_accept_rate_tv(1, B, g, V, binding.BF16, d_, t_, keep, None, acc, emask, tau, ws_t)
        ev[4].record()
        return ev

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    for w in (ws_s, ws_a, ws_v, ws_t):
        assert binding.dspark_get_device_status(w) == 0
    n_rej = int((nacc < Lout).sum().item())
    n_ver = int(Lout.sum().item())

    names = ["schedule", "sample", "verify", "tv"]
    per = {n: [] for n in names}
    step_ms = []
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.wait_first()
        wall0 = time.perf_counter()
        launches0 = binding.dspark_kernel_launches()
        evs = []
        for _ in range(args.steps):
            flush.zero_()
            evs.append(step())
        launches = binding.dspark_kernel_launches() - launches0  # the library's own kernels, counted by it
        torch.cuda.synchronize()
        wall1 = time.perf_counter()
        wall = wall1 - wall0
        time.sleep(0.25)  # let the sample that covers the end of the window arrive
    for ev in evs:
        for k, n in enumerate(names):
            per[n].append(ev[k].elapsed_time(ev[k + 1]))
        step_ms.append(ev[0].elapsed_time(ev[4]))
    t_step = shard.max_over_ranks(sum(step_ms) / len(step_ms), pg, dev)
    value = shard.job_throughput(B * g, world, t_step * 1e-3)

    # e2e: the same step through the C ABI with host inputs copied in and results read back.
    # Serving-style pipeline: while step k computes, a copy stream uploads step k+1's inputs from
    # pinned host memory into the other of two device buffer sets (events keep a set from being
    # overwritten before its step is done).  A window opens on the compute stream once everything
    # before it has finished (the first upload waits for it) and closes after the last step's
    # read-back, so it holds exactly its steps' copies and compute.  The inputs (two sets larger
    # than L2) need no flush between steps.  Three windows give the spread.
    pin = {k: v.cpu().pin_memory() for k, v in (("base", base), ("target", target), ("conf", conf), ("anchor", anchor))}
    dsets = [{k: torch.empty_like(v) for k, v in (("base", base), ("target", target), ("conf", conf), ("anchor", anchor))}
             for _ in range(2)]
    outs = [tok, nacc, corr, acc, emask, tau, Lout]
    hout = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = sum(o.numel() * o.element_size() for o in outs)
    comp = torch.cuda.current_stream(dev)
    copy_s = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]  # a set's inputs have arrived
    free = [torch.cuda.Event() for _ in range(2)]   # a set's step has finished with it

    def upload(it):
        st_ = it % 2
        with torch.cuda.stream(copy_s):
            if it >= 2:
                copy_s.wait_event(free[st_])
            for k in pin:
                dsets[st_][k].copy_(pin[k], non_blocking=True)
            ready[st_].record(copy_s)

    def pipeline(n):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        copy_s.wait_event(e0)
        upload(0)
        for it in range(n):
            if it + 1 < n:
                upload(it + 1)
            st_ = it % 2
            comp.wait_event(ready[st_])
            dset = dsets[st_]
            step((dset["base"], dset["target"], dset["conf"], dset["anchor"]))
            free[st_].record(comp)
            for o, h in zip(outs, hout):
                h.copy_(o, non_blocking=True)
        e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    e2e_steps = max(1, min(args.steps, E2E_STEPS))
    pipeline(max(args.warmup, 3))
    e2e_ms = sorted(pipeline(e2e_steps) for _ in range(3))
    t_e2e = shard.max_over_ranks(e2e_ms[1], pg, dev)

    avg = {n: sum(v) / len(v) for n, v in per.items()}
    algo = algorithmic_bytes(wl, n_rej, n_ver)
    peak, peak_kind = peaks()
    dom = max(["sample", "verify", "tv"], key=lambda n: avg[n])
    achieved = algo[dom] / (avg[dom] * 1e-3) / 1e9
    kernels = {n: {"ms": round(avg[n], 5), "bytes": algo[n],
                   "gbs": round(algo[n] / (avg[n] * 1e-3) / 1e9, 1),
                   "frac_of_peak": round(algo[n] / (avg[n] * 1e-3) / 1e9 / peak, 4)} for n in names}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "draft tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(t_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": args.workload, "B": B, "gamma": g, "V": V, "r": wl.r, "T": wl.T, "budget": budget,
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed (256 MB write) before each step; per-step CUDA events exclude the flush",
                   "step": "schedule + sample + verify + tv(eval_mask, tau)"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": profiled_traffic(dom), "algorithmic_bytes": algo[dom]},
        "kernels": kernels,
        "n_rejected": n_rej,
        "e2e": {"value": round(shard.job_throughput(B * g, world, t_e2e * 1e-3), 1), "unit": "draft tokens/s",
                "ms_per_step": round(t_e2e, 4), "ms_per_step_windows": [round(x, 4) for x in e2e_ms],
                "steps_per_window": e2e_steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "verified_tokens_per_s": round(shard.job_throughput(n_ver, world, (avg["schedule"] + avg["verify"]) * 1e-3), 1),
        "gpu_launches": launches,
        "clocks": clk.summary(wall0, wall1 + 0.2),
        "wall_s_timed": round(wall, 3),
    }
    # outside the step: the throughput-aware prefix choice on the same confidences (a per-request
    # causal search; one launch), timed alone with CUDA events after the step's timing
    sps = torch.clamp(1.0 - 0.05 * torch.arange(g + 1, dtype=torch.float32, device=dev), min=0.05)
    ell = torch.empty(B, dtype=torch.int32, device=dev)
    for _ in range(3):
        binding.dspark_theta_schedule(B, g, conf, sps, ell)
    th_ms = []
    for _ in range(200):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()  # the device is busy while the launch below is submitted: the events time the kernel
        e0.record()
        binding.dspark_theta_schedule(B, g, conf, sps, ell)
        e1.record()
        th_ms.append((e0, e1))
    torch.cuda.synchronize()
    th_us = sorted(a.elapsed_time(b_) * 1e3 for a, b_ in th_ms)
    # teacher-forced block logits of the same batch (the drafted tokens as the true ones), fp32 out
    zt = torch.empty((B, g, V), dtype=torch.float32, device=dev)
    ws_z = binding.workspace(binding.dspark_markov_block_logits_workspace_size(p), dev)
    for _ in range(3):
        binding.dspark_markov_block_logits(p, base, W1, W2, anchor, tok, zt, ws_z)
    bl = []
    for _ in range(50):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        e0.record()
        binding.dspark_markov_block_logits(p, base, W1, W2, anchor, tok, zt, ws_z)
        e1.record()
        bl.append((e0, e1))
    torch.cuda.synchronize()
    bl_us = sorted(a.elapsed_time(b_) * 1e3 for a, b_ in bl)[len(bl) // 2]
    bl_bytes = B * g * V * base.element_size() + V * wl.r * W2.element_size() + B * g * V * 4
    # the training-side L1 term on this step's accept rates (one block)
    l1b = torch.empty_like(acc)
    l1s = torch.empty(2, dtype=torch.float64, device=dev)
    l1t = []
    for _ in range(50):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        e0.record()
        binding.dspark_tv_l1_loss(1, B, g, acc, emask, 4.0, l1b, l1s)
        e1.record()
        l1t.append((e0, e1))
    torch.cuda.synchronize()
    l1_us = sorted(a.elapsed_time(b_) * 1e3 for a, b_ in l1t)[len(l1t) // 2]
    # the draft sampler with a final-logit softcap (s tanh(b / s) on every base logit; s = 30): the
    # same call as the step's, on the sampler that supports the cap
    pc = api.make_params(base, W1, wl.T, wl.seed, softcap=30.0)
    ws_c = binding.workspace(binding.dspark_sample_workspace_size(pc), dev)
    tok_c = torch.empty_like(tok)
    lse_c = torch.empty((B, g), device=dev)
    zat_c = torch.empty((B, g), device=dev)
    for _ in range(3):
        binding.dspark_markov_sample_block(pc, base, W1, W2, anchor, tok_c, lse_c, zat_c, ws_c)
    sc = []
    for _ in range(20):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        e0.record()
        binding.dspark_markov_sample_block(pc, base, W1, W2, anchor, tok_c, lse_c, zat_c, ws_c)
        e1.record()
        sc.append((e0, e1))
    torch.cuda.synchronize()
    sc_us = sorted(a.elapsed_time(b_) * 1e3 for a, b_ in sc)[len(sc) // 2]
    line["extras"] = {"tv_l1_loss_us": round(l1_us, 2),
                      "sample_softcap_us": round(sc_us, 2),
                      "sample_softcap_frac_of_peak": round(algo["sample"] / (sc_us * 1e-6) / 1e9 / peak, 4),
                      "sample_softcap": "the step's sampling call with softcap 30 (tanh on every base logit), median "
                                        "of 20 launches; the same algorithmic bytes as the step's sampler",
                      "theta_schedule_us": round(th_us[len(th_us) // 2], 2),
                      "theta_schedule": f"median of 200 launches over B={B} requests, gamma={g}; not part of the step",
                      "block_logits_us": round(bl_us, 2),
                      "block_logits_frac_of_peak": round(bl_bytes / (bl_us * 1e-6) / 1e9 / peak, 4),
                      "block_logits": f"teacher-forced z [B,gamma,V] fp32 of the batch, median of 50 launches, "
                                      f"{bl_bytes} algorithmic bytes (base + W2 read, z written); not part of the step"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_baseline(host, wl_name=args.workload, T=wl.T, budget=wl.budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
