"""Benchmark: tree-packed attention forward + backward on one GB300.

A step is one tree_attn_fwd plus the backward over one synthetic batch (the
whole hot path: the plan is built once per batch, outside the timed region, as
the pages build it once per forward on the host). The backward is issued as its
two phases, tree_attn_bwd_dq and tree_attn_bwd_dkdv (the two launches
tree_attn_bwd makes), so that CUDA events time each of the three kernels; the
``roofline`` object is for the slowest of them. The headline
workload is the packed batch of 32 GRPO-shaped tries, 131,072 tokens, 64 q
heads / 8 kv heads, head_dim 128, bf16.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5] [--impl reference]

Prints one JSON line. ``value`` is visible-pair TFLOP/s of fwd+bwd
((4 + 10) * D * Hq * visible pairs per step), summed over ranks; inputs are
resident in HBM and larger than L2, and L2 is also flushed between steps.
``e2e`` is the same metric with host (pinned) buffers: every step's inputs are
copied host->device and all its outputs device->host inside the timed region
(host wall clock from the first copy to the last), with the copies of
neighbouring steps overlapping the compute on separate streams.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-attn fwd+bwd visible-pair TFLOP/s and tokens/s on 1 GB300; % of bf16 peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return FALLBACK_PEAKS, "fallback"


# DRAM bytes per launch from an ncu capture, kept only while the kernel's
# sources still hash to what they were when the counters were taken.
KERNEL_SOURCES = {
    "tree_rope_kernel": ("rope.cu",),
    "tree_attn_fwd_sm103": ("fwd_sm103.cu", "sm103_ptx.cuh"),
    "tree_attn_bwd_dq_sm103": ("bwd_sm103.cu", "sm103_ptx.cuh"),
    "tree_attn_bwd_dkdv_sm103": ("bwd_sm103.cu", "sm103_ptx.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    import hashlib

    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "tree_packed_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(workload: str, kernel: str):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload, {}).get(kernel)
    except OSError:
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


def _dist(backend: str = "nccl"):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group(backend)
        return dist, dist.get_rank(), ws
    return None, 0, 1


def max_over_ranks(x: float, dist, device="cpu") -> float:
    """The largest of every rank's x: a job of replicas is as slow as its slowest one."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, work_per_replica: float, ms: float) -> float:
    """Units per second over all replicas, each doing work_per_replica in (max) ms."""
    return world * work_per_replica / (ms * 1e-3)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_sample(workload_index: int, min_seconds: float = 10.0):
    """Time the CPU oracle (fp64) on a bounded sample of the workload.

    The sample is whole tries of the workload (the subtree of the first root,
    then the next, ...) with one kv-head group each (hq/hkv q heads, one kv
    head): full forward and backward, until at least ``min_seconds`` of CPU
    work or every trie has been done. Returns (visible-pair TFLOP/s,
    tokens/s, description, threads, seconds).
    """
    import numpy as np
    import torch

    import treegen
    from oracle import attention as A
    from oracle import mask as M

    w = treegen.workload(workload_index)
    parents = np.asarray(w.parents)
    roots = np.flatnonzero(parents == -1)

    def root_of(s):
        while parents[s] != -1:
            s = parents[s]
        return s

    owner = np.array([root_of(s) for s in range(len(parents))])
    g = w.hq // w.hkv
    threads = len(os.sched_getaffinity(0))
    torch.set_num_threads(threads)
    flops = 0.0
    tokens = 0
    done = 0
    elapsed = 0.0
    for t, r in enumerate(roots):
        members = np.flatnonzero(owner == r).tolist()
        remap = {s: n for n, s in enumerate(members)}
        sub_p = np.array([-1 if parents[s] == -1 else remap[parents[s]] for s in members], np.int32)
        sub_l = np.asarray(w.lengths)[members].astype(np.int32)
        n = int(sub_l.sum())
        q, k, v, do = treegen.draw_tensors(n, g, 1, w.head_dim, w.dtype, seed=t)
        pvis = M.TrieView(sub_p, sub_l).visible_count()
        t0 = time.perf_counter()
        A.forward(q, k, v, sub_p, sub_l)
        A.backward(q, k, v, do, sub_p, sub_l)
        elapsed += time.perf_counter() - t0
        flops += 14.0 * w.head_dim * g * pvis
        tokens += n
        done += 1
        if elapsed >= min_seconds:
            break
    desc = (f"{done} of {len(roots)} tries of the workload ({tokens} tokens) x one kv group "
            f"({g} q heads, 1 kv head), fp64 forward + backward")
    return flops / elapsed / 1e12, tokens / elapsed, desc, threads, elapsed


def reference_arm(args):
    """The CPU oracle as the reference arm: each step is the bounded sample above."""
    dist, rank, world = None, int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import treegen

    w = treegen.workload(args.workload)
    vals, toks, times = [], [], []
    desc, threads = "", 0
    per_step = min(10.0, 150.0 / max(1, args.steps + args.warmup))  # whole run: a few minutes
    for _ in range(args.warmup):
        cpu_oracle_sample(args.workload, per_step)
    for _ in range(args.steps):
        v, t, desc, threads, dt = cpu_oracle_sample(args.workload, per_step)
        vals.append(v)
        toks.append(t)
        times.append(dt)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "tokens_per_s": statistics.mean(toks),
        "config": {"workload": w.name, "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def time_workload(index: int, steps: int, warmup: int, dev, rank: int, clock_gpu=None):
    """Build the plan of workload ``index``, draw its inputs on the device and
    time ``steps`` steps (forward, then the backward's two phases) with CUDA
    events around each kernel, L2 flushed between steps. Returns a dict of the
    per-step event times and what the end-to-end leg needs."""
    import torch

    import treegen
    import tree_packed_attention_gb300 as tpa

    w = treegen.workload(index)
    N, hq, hkv, D = w.num_tokens, w.hq, w.hkv, w.head_dim
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    t0 = time.perf_counter()
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    plan_ms = 1e3 * (time.perf_counter() - t0)
    plan.to_device()

    # Seeded synthetic inputs, N(0,1), drawn on the device (one generator per rank).
    gen = torch.Generator(device=dev).manual_seed(1000 + rank)
    q = torch.randn(N, hq, D, generator=gen, device=dev, dtype=torch.float32).to(tdt)
    k = torch.randn(N, hkv, D, generator=gen, device=dev, dtype=torch.float32).to(tdt)
    v = torch.randn(N, hkv, D, generator=gen, device=dev, dtype=torch.float32).to(tdt)
    do = torch.randn(N, hq, D, generator=gen, device=dev, dtype=torch.float32).to(tdt)
    o = torch.empty_like(q)
    lse = torch.empty(hq, N, dtype=torch.float32, device=dev)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws = torch.empty(tpa.tree_attn_bwd_workspace_bytes(plan, hq, D, tdt), dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(warmup):
        tpa.tree_attn_fwd(plan, q, k, v, out=o, lse=lse)
        tpa.tree_attn_bwd(plan, do, q, k, v, o, lse, workspace=ws, out=(dq, dk, dv))
    tpa.tree_status_sync()

    # The timed step runs the backward as its two phases (exactly what
    # tree_attn_bwd launches) so that each kernel gets its own events.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    torch.cuda.synchronize()
    clocks = ClockSampler(clock_gpu) if clock_gpu is not None else None
    if clocks:
        clocks.__enter__()
    for st in range(steps):
        flush.zero_()  # L2 flush between timed steps (outside the events)
        ev[st][0].record(stream)
        tpa.tree_attn_fwd(plan, q, k, v, out=o, lse=lse)
        ev[st][1].record(stream)
        tpa.tree_attn_bwd_dq(plan, do, q, k, v, o, lse, ws, out=dq)
        ev[st][2].record(stream)
        tpa.tree_attn_bwd_dkdv(plan, do, q, k, v, lse, ws, out=(dk, dv))
        ev[st][3].record(stream)
    torch.cuda.synchronize()
    if clocks:
        clocks.__exit__(None, None, None)
    tpa.tree_status_sync()
    return {
        "w": w, "plan": plan, "plan_ms": plan_ms, "pvis": plan.info["visible_pairs"],
        "tensors": (q, k, v, do, o, lse, dq, dk, dv, ws), "clocks": clocks,
        "fwd_ms": [e[0].elapsed_time(e[1]) for e in ev],
        "dq_ms": [e[1].elapsed_time(e[2]) for e in ev],
        "kv_ms": [e[2].elapsed_time(e[3]) for e in ev],
    }


def kernel_table(r):
    """Mean event time of each kernel and the FLOPs its outputs need per
    visible pair and q head (fwd: S, PV; dQ: S, dP, dS K; dK/dV: S^T, dP^T,
    P^T dO, dS^T Q)."""
    w, pvis = r["w"], r["pvis"]
    D, hq = w.head_dim, w.hq
    return {
        "tree_attn_fwd_sm103": (statistics.mean(r["fwd_ms"]), 4.0 * D * hq * pvis),
        "tree_attn_bwd_dq_sm103": (statistics.mean(r["dq_ms"]), 6.0 * D * hq * pvis),
        "tree_attn_bwd_dkdv_sm103": (statistics.mean(r["kv_ms"]), 8.0 * D * hq * pvis),
    }


def workload_summary(r, peak):
    """fwd / bwd / fwd+bwd visible-pair TFLOP/s and fractions of the bf16 peak
    for one timed workload (metric accounting: 4*D and 10*D per pair and head)."""
    w, pvis = r["w"], r["pvis"]
    D, hq = w.head_dim, w.hq
    fwd = statistics.mean(r["fwd_ms"])
    bwd = statistics.mean(a + b for a, b in zip(r["dq_ms"], r["kv_ms"]))
    f_tf = 4.0 * D * hq * pvis / (fwd * 1e-3) / 1e12
    b_tf = 10.0 * D * hq * pvis / (bwd * 1e-3) / 1e12
    t_tf = 14.0 * D * hq * pvis / ((fwd + bwd) * 1e-3) / 1e12
    return {
        "workload": w.name, "tokens": w.num_tokens, "hq": hq, "hkv": w.hkv, "head_dim": D,
        "visible_pairs": pvis, "ms_per_step": fwd + bwd,
        "fwd_bwd": {"tflops": t_tf, "frac": t_tf / peak},
        "fwd": {"ms": fwd, "tflops": f_tf, "frac": f_tf / peak},
        "bwd": {"ms": bwd, "tflops": b_tf, "frac": b_tf / peak},
        "kernels": {n: {"ms": t, "tflops_algorithmic": f / (t * 1e-3) / 1e12}
                    for n, (t, f) in kernel_table(r).items()},
    }


def gpu_arm(args):
    import torch

    import tree_packed_attention_gb300 as tpa

    dist, rank, world = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_kind = _peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    # Secondary workloads first (their tensors are freed before the headline's).
    extras = []
    for idx in [int(x) for x in args.extra_workloads.split(",") if x.strip()]:
        if idx == args.workload:
            continue
        r = time_workload(idx, max(3, min(args.steps, 10)), args.warmup, dev, rank)
        for key in ("fwd_ms", "dq_ms", "kv_ms"):
            r[key] = [max_over_ranks(statistics.mean(r[key]), dist, dev)]
        extras.append(workload_summary(r, peak))
        del r
        torch.cuda.empty_cache()

    if dist:
        dist.barrier()
    r = time_workload(args.workload, args.steps, args.warmup, dev, rank, clock_gpu=local)
    if dist:
        dist.barrier()
    w, plan, plan_ms, pvis, clocks = r["w"], r["plan"], r["plan_ms"], r["pvis"], r["clocks"]
    q, k, v, do, o, lse, dq, dk, dv, ws = r["tensors"]
    N, hq, hkv, D = w.num_tokens, w.hq, w.hkv, w.head_dim
    flops_fwd = 4.0 * D * hq * pvis
    flops_bwd = 10.0 * D * hq * pvis
    fwd_ms, dq_ms, kv_ms = r["fwd_ms"], r["dq_ms"], r["kv_ms"]
    bwd_ms = [a + b for a, b in zip(dq_ms, kv_ms)]
    step_ms = statistics.mean(f + b for f, b in zip(fwd_ms, bwd_ms))
    step_ms = max_over_ranks(step_ms, dist, dev)
    value = whole_job_rate(world, flops_fwd + flops_bwd, step_ms) / 1e12
    tokens_s = whole_job_rate(world, N, step_ms)

    # End to end through the public API with pinned host buffers. Every step
    # copies its inputs host->device, runs forward and backward, and copies
    # every output device->host; three streams let step s+1's inputs and step
    # s-1's outputs cross the host link while step s computes (two device
    # buffer sets, events order the reuse of each set).
    hq_pin = [x.cpu().pin_memory() for x in (q, k, v, do)]
    out_pin = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (o, lse, dq, dk, dv)]
               for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in hq_pin)
    d2h = sum(x.numel() * x.element_size() for x in out_pin[0])
    e2e_steps = max(3, min(args.steps, 10))
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    dev_in = [[torch.empty_like(x) for x in (q, k, v, do)] for _ in range(2)]
    dev_out = [[torch.empty_like(x) for x in (o, lse, dq, dk, dv)] for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set b landed
    ev_run = [torch.cuda.Event() for _ in range(2)]   # compute on set b done
    ev_out = [torch.cuda.Event() for _ in range(2)]   # outputs of set b copied out
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_run[b])  # the compute that read this set is done
            for dst, src in zip(dev_in[b], hq_pin):
                dst.copy_(src, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[b])
            if used[b]:
                s_run.wait_event(ev_out[b])  # this set's previous outputs are out
            qq, kk, vv, dd = dev_in[b]
            oo, ll, gq, gk, gv = dev_out[b]
            tpa.tree_attn_fwd(plan, qq, kk, vv, out=oo, lse=ll, stream=s_run)
            tpa.tree_attn_bwd(plan, dd, qq, kk, vv, oo, ll, workspace=ws, out=(gq, gk, gv),
                              stream=s_run)
            ev_run[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[b])
            for dst, src in zip(out_pin[b], dev_out[b]):
                dst.copy_(src, non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(2):  # warm both buffer sets
        e2e_step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_e2e = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_ms = 1e3 * (time.perf_counter() - t_e2e) / e2e_steps
    tpa.tree_status_sync()
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = whole_job_rate(world, flops_fwd + flops_bwd, e2e_ms) / 1e12

    bwd_mean = statistics.mean(bwd_ms)
    fwd_mean = statistics.mean(fwd_ms)
    bwd_tf = flops_bwd / (bwd_mean * 1e-3) / 1e12
    fwd_tf = flops_fwd / (fwd_mean * 1e-3) / 1e12
    kernels = kernel_table(r)
    top = max(kernels, key=lambda n: kernels[n][0])
    top_ms, top_flops = kernels[top]
    top_tf = top_flops / (top_ms * 1e-3) / 1e12
    traffic = _traffic(w.name, top)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, t_cpu, desc, threads, dt = cpu_oracle_sample(args.workload)
        cpu = {"value": v_cpu, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc,
               "tokens_per_s": t_cpu, "seconds": dt}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "tokens": N, "hq": hq, "hkv": hkv, "head_dim": D,
                       "visible_pairs": pvis, "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2, and L2 flushed between steps"},
            "tokens_per_s": tokens_s,
            "fraction_of_bf16_peak": value / world / peak,
            "fwd": {"ms": fwd_mean, "tflops": fwd_tf, "frac": fwd_tf / peak, "launches": 1},
            "bwd": {"ms": bwd_mean, "tflops": bwd_tf, "frac": bwd_tf / peak, "launches": 2},
            "kernels": {n: {"ms": t, "tflops_algorithmic": f / (t * 1e-3) / 1e12}
                        for n, (t, f) in kernels.items()},
            "plan_build_ms": plan_ms,
            "roofline": {"bound": "tensor", "kernel": top, "achieved": top_tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": top_tf / peak,
                         "peak_source": f"{peak_kind} bf16 dense (burst)", "traffic": traffic},
            "clocks": clocks.summary(),
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": 3 * args.steps,
            "cpu_baseline": cpu,
            # the other tree-shaped workloads, timed the same way in this run
            # (fewer steps), so their fractions sit in the same record
            "workloads": extras,
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def rope_arm(args):
    """--op rope: tree RoPE (position ids of eq. 9) applied in place to the
    workload's q and k, bf16, one GPU. HBM-bound: every element is read and
    written once, so the figure is algorithmic bytes / event time against the
    measured copy bandwidth."""
    import torch

    import treegen
    import tree_packed_attention_gb300 as tpa

    torch.cuda.set_device(0)
    w = treegen.workload(args.workload)
    N, hq, hkv, D = w.num_tokens, w.hq, w.hkv, w.head_dim
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    gen = torch.Generator(device="cuda").manual_seed(0)
    q = torch.randn(N, hq, D, device="cuda", generator=gen).to(torch.bfloat16)
    k = torch.randn(N, hkv, D, device="cuda", generator=gen).to(torch.bfloat16)
    stream = torch.cuda.current_stream()
    plan.to_device(stream)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    nbytes = 2 * (q.numel() + k.numel()) * q.element_size()  # read and write each element once
    for _ in range(args.warmup):
        tpa.tree_rope_qk(plan, q, k)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(0) as clocks:
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            tpa.tree_rope_qk(plan, q, k)  # q and k in one launch
            b.record(stream)
        torch.cuda.synchronize()
    tpa.tree_status_sync()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, kind = _peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    traffic = _traffic(w.name, "tree_rope_kernel")
    print(json.dumps({
        "metric": "tree RoPE at eq. 9 position ids, q and k in place, GB/s on 1 GB300", "value": gbs,
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "tokens": N, "hq": hq, "hkv": hkv, "head_dim": D,
                   "l2": "inputs larger than L2, and L2 flushed between steps"},
        "roofline": {"bound": "hbm", "kernel": "tree_rope_kernel", "achieved": gbs, "peak": peak,
                     "unit": "GB/s", "frac": gbs / peak, "peak_source": f"{kind} copy bandwidth",
                     "traffic": traffic},  # the step's one launch (q and k)
        "bytes_per_step": nbytes, "clocks": clocks.summary(), "gpu_launches": args.steps,
    }))


def conv_arm(args):
    """--op conv: the tree-correct causal conv (App. A.3) forward and backward
    on the workload's tokens, bf16, K = 4, SiLU, C = --channels. Memory-bound:
    the figure is the algorithmic bytes (forward reads x and writes y; the
    backward reads x and dy and writes dx) over the CUDA-event time."""
    import torch

    import treegen
    import tree_packed_attention_gb300 as tpa

    torch.cuda.set_device(0)
    w = treegen.workload(args.workload)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N, C, K = plan.num_tokens, args.channels, 4
    gen = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn(N, C, device="cuda", generator=gen).to(torch.bfloat16)
    dy = torch.randn(N, C, device="cuda", generator=gen).to(torch.bfloat16)
    wt = torch.randn(C, K, device="cuda", generator=gen) * 0.5
    b = torch.randn(C, device="cuda", generator=gen)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    y = torch.empty_like(x)
    for _ in range(args.warmup):
        tpa.tree_conv_fwd(plan, x, wt, b, out=y)
        tpa.tree_conv_bwd(plan, x, wt, b, dy)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(0) as clocks:
        for e in ev:
            flush.zero_()
            e[0].record(stream)
            tpa.tree_conv_fwd(plan, x, wt, b, out=y)
            e[1].record(stream)
            tpa.tree_conv_bwd(plan, x, wt, b, dy)
            e[2].record(stream)
        torch.cuda.synchronize()
    tpa.tree_status_sync()
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    row = C * x.element_size()
    fwd_bytes, bwd_bytes = 2 * N * row, 3 * N * row
    gbs = (fwd_bytes + bwd_bytes) / ((fwd_ms + bwd_ms) * 1e-3) / 1e9
    peaks, kind = _peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    print(json.dumps({
        "metric": "tree-correct causal conv (K=4, SiLU) forward+backward, algorithmic GB/s on 1 GB300",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": fwd_ms + bwd_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "tokens": N, "channels": C, "kernel_size": K,
                   "l2": "inputs larger than L2, and L2 flushed between steps"},
        "fwd": {"ms": fwd_ms, "gbs": fwd_bytes / (fwd_ms * 1e-3) / 1e9},
        "bwd": {"ms": bwd_ms, "gbs": bwd_bytes / (bwd_ms * 1e-3) / 1e9},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_source": f"{kind} copy bandwidth", "traffic": None},
        "clocks": clocks.summary(), "gpu_launches": 5 * args.steps,
    }))


def ce_arm(args):
    """--op ce: the fused weighted next-token cross-entropy (§3.1 eq. 3-5) with its
    gradient, bf16 logits [N, V] of the workload (default 6: the packed shape at
    32,768 tokens) and V = --vocab, lambda = g/K. HBM-bound: the figure is the
    algorithmic bytes (logits read once, dlogits written once) over the
    CUDA-event time; the kernel reads each row a second time from L2."""
    import torch

    import treegen
    import tree_packed_attention_gb300 as tpa

    torch.cuda.set_device(0)
    w = treegen.workload(args.workload)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N, V = plan.num_tokens, args.vocab
    gen = torch.Generator(device="cuda").manual_seed(0)
    z = torch.empty(N, V, dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, N, 4096):  # drawn in slices to bound the fp32 temporary
        r1 = min(N, r0 + 4096)
        z[r0:r1] = (torch.randn(r1 - r0, V, device="cuda", generator=gen) * 3).to(torch.bfloat16)
    tokens = torch.randint(0, V, (N,), device="cuda", generator=gen, dtype=torch.int32)
    lam = torch.as_tensor(tpa.tree_weights(plan), device="cuda")
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        loss, row_loss, dz = tpa.tree_weighted_ce(plan, z, tokens, lam)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    with ClockSampler(0) as clocks:
        for e in ev:
            flush.zero_()
            e[0].record(stream)
            loss, row_loss, dz = tpa.tree_weighted_ce(plan, z, tokens, lam)
            e[1].record(stream)
        torch.cuda.synchronize()
    tpa.tree_status_sync()
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    algo = 2 * N * V * z.element_size()
    gbs = algo / (ms * 1e-3) / 1e9
    peaks, kind = _peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    print(json.dumps({
        "metric": "fused weighted tree cross-entropy (loss + dlogits), algorithmic GB/s on 1 GB300",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "tokens": N, "vocab": V, "weights": "g/K",
                   "l2": "inputs larger than L2, and L2 flushed between steps"},
        "tokens_per_s": N / (ms * 1e-3), "loss": float(loss),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_source": f"{kind} copy bandwidth", "traffic": None},
        "clocks": clocks.summary(), "gpu_launches": 2 * args.steps,
    }))


def gateway_pieces(parents, lengths, part_of, plan):
    """The pieces of a node-boundary partition with their gateways (App. B.2-B.3):
    per piece its segments renumbered as a trie of its own, its tokens (global
    DFS indices), and its gateway: the parent piece's gateway followed by the
    parent piece's DFS tokens up to the end of the cut node, visible where they
    lie on the chain from the parent piece's root down to the cut node (the
    parent's own gateway keeps the visibility it had for the parent)."""
    order = [int(s) for s in plan.field("dfs_order")]
    start = plan.field("seg_start")
    tok = {s: range(int(start[s]), int(start[s]) + int(lengths[s])) for s in order}
    out, ids = {}, []
    for s in order:
        if part_of[s] not in ids:
            ids.append(part_of[s])
    for pid in ids:
        segs = [s for s in order if part_of[s] == pid]
        local = {s: n for n, s in enumerate(segs)}
        lp = [local[parents[s]] if parents[s] >= 0 and part_of[parents[s]] == pid else -1 for s in segs]
        gw, vis = [], []
        root = segs[0]
        if parents[root] >= 0:
            nc = parents[root]
            pp = out[part_of[nc]]
            chain, a = set(), nc
            while a >= 0 and part_of[a] == part_of[nc]:
                chain.add(a)
                a = parents[a]
            gw, vis = list(pp["gw"]), list(pp["vis"])
            for s in pp["segs"]:
                gw.extend(tok[s])
                vis.extend([s in chain] * len(tok[s]))
                if s == nc:
                    break
        out[pid] = {"segs": segs, "parents": lp, "lengths": [int(lengths[s]) for s in segs],
                    "tokens": [t for s in segs for t in tok[s]], "gw": gw, "vis": vis}
    return [out[pid] for pid in ids]


def gateway_arm(args):
    """--op gateway: partition-gateway attention (App. B.2-B.5). The workload's
    trie (default 4: agentic, 65,536 tokens, 16 heads) cut by tree_partition into
    pieces of at most --cap tokens; one step is the forward and backward of every
    piece over its own keys and its gateway (its ancestors' cached keys), with
    the gateway gradients accumulated in fp32. The figure counts each piece's
    visible pairs, its own plus its rows times its visible gateway keys, which
    together are the whole trie's, at 4·D (forward) + 10·D (backward) flops per
    pair and q head; the whole trie in one call is timed the same way beside it."""
    import torch

    import treegen
    import tree_packed_attention_gb300 as tpa

    torch.cuda.set_device(0)
    w = treegen.workload(args.workload)
    whole = tpa.tree_plan_build(w.parents, w.lengths)
    N, hq, hkv, D = w.num_tokens, w.hq, w.hkv, w.head_dim
    r = tpa.tree_partition(whole, args.cap)
    part = [int(x) for x in r["part_of_segment"]]
    parents = [int(x) for x in w.parents]
    Xs = gateway_pieces(parents, w.lengths, part, whole)
    gen = torch.Generator(device="cuda").manual_seed(0)
    q, do = (torch.randn(N, hq, D, device="cuda", generator=gen).to(torch.bfloat16) for _ in range(2))
    k, v = (torch.randn(N, hkv, D, device="cuda", generator=gen).to(torch.bfloat16) for _ in range(2))
    runs, pairs = [], 0
    for X in Xs:
        t = torch.as_tensor(X["tokens"], dtype=torch.long, device="cuda")
        g = torch.as_tensor(X["gw"], dtype=torch.long, device="cuda")
        plan = tpa.tree_plan_build_partition(X["parents"], X["lengths"], X["vis"])
        P = plan.info["past_len"]
        acc = [torch.zeros(P, hkv, D, dtype=torch.float32, device="cuda") for _ in range(2)]
        ws = torch.empty(max(tpa.tree_attn_bwd_workspace_bytes(plan, hq, D, torch.bfloat16), 16),
                         dtype=torch.uint8, device="cuda")
        runs.append((plan, q[t].contiguous(), k[t].contiguous(), v[t].contiguous(), do[t].contiguous(),
                     k[g].contiguous(), v[g].contiguous(), acc, ws))
        pairs += int(plan.info["visible_pairs"]) + len(X["tokens"]) * int(plan.info["past_visible"])
    assert pairs == int(whole.info["visible_pairs"]), (pairs, whole.info["visible_pairs"])

    def step_pieces():
        for plan, qp, kp, vp, dop, pk, pv, acc, ws in runs:
            acc[0].zero_()
            acc[1].zero_()
            o, lse = tpa.tree_attn_fwd_gateway(plan, qp, kp, vp, pk, pv)
            tpa.tree_attn_bwd_gateway(plan, dop, qp, kp, vp, pk, pv, o, lse, acc[0], acc[1], workspace=ws)

    ws_whole = torch.empty(tpa.tree_attn_bwd_workspace_bytes(whole, hq, D, torch.bfloat16), dtype=torch.uint8,
                           device="cuda")

    def step_whole():
        o, lse = tpa.tree_attn_fwd(whole, q, k, v)
        tpa.tree_attn_bwd(whole, do, q, k, v, o, lse, workspace=ws_whole)

    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for e in ev:
            flush.zero_()
            e[0].record(stream)
            fn()
            e[1].record(stream)
        torch.cuda.synchronize()
        tpa.tree_status_sync()
        return statistics.mean(e[0].elapsed_time(e[1]) for e in ev)

    with ClockSampler(0) as clocks:
        ms = timed(step_pieces)
    ms_whole = timed(step_whole)
    flops = 14.0 * D * hq * pairs
    tf = flops / (ms * 1e-3) / 1e12
    peaks, kind = _peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    print(json.dumps({
        "metric": "partition-gateway attention fwd+bwd over every piece, visible-pair TFLOP/s on 1 GB300",
        "value": tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "tokens": N, "hq": hq, "hkv": hkv, "head_dim": D, "cap": args.cap,
                   "pieces": len(Xs), "gateway_keys": int(sum(len(X["gw"]) for X in Xs)),
                   "visible_pairs": pairs, "l2": "L2 flushed between steps"},
        "whole_trie": {"ms": ms_whole, "tflops": flops / (ms_whole * 1e-3) / 1e12},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                     "peak_source": f"{kind} bf16 dense (burst)", "traffic": None},
        "clocks": clocks.summary(), "gpu_launches": 3 * len(Xs) * args.steps,
    }))


def gdn_arm(args):
    """--op gdn: the Gated DeltaNet forward with tree state routing (eq. 10,
    App. A.2) over the workload's trie, bf16 q/k/v, --gdn-heads query/key heads
    and twice as many value heads (head_dim 128; a Qwen3-Next-shaped layer).
    Bound by the FMA pipe: the figure is 3 * 128 * 128 fused multiply-adds per
    token and value head (the key product, the state update, the query
    product) over the CUDA-event time, against 152 SMs x 128 FP32 lanes x 2
    flops x the sampled SM clock."""
    import torch

    import treegen
    import tree_packed_attention_gb300 as tpa

    torch.cuda.set_device(0)
    w = treegen.workload(args.workload)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N = plan.num_tokens
    hk = args.gdn_heads
    hv = 2 * hk
    gen = torch.Generator(device="cuda").manual_seed(0)

    def unit(x):
        return x / x.norm(dim=-1, keepdim=True)

    q = unit(torch.randn(N, hk, 128, device="cuda", generator=gen)).to(torch.bfloat16)
    k = unit(torch.randn(N, hk, 128, device="cuda", generator=gen)).to(torch.bfloat16)
    v = torch.randn(N, hv, 128, device="cuda", generator=gen).to(torch.bfloat16)
    g = -0.5 * torch.rand(N, hv, device="cuda", generator=gen)
    beta = torch.rand(N, hv, device="cuda", generator=gen)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        o, states = tpa.tree_gdn_fwd(plan, q, k, v, g, beta)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    with ClockSampler(0) as clocks:
        for e in ev:
            flush.zero_()
            e[0].record(stream)
            o, states = tpa.tree_gdn_fwd(plan, q, k, v, g, beta)
            e[1].record(stream)
        torch.cuda.synchronize()
    tpa.tree_status_sync()
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    flops = 2.0 * 3 * 128 * 128 * N * hv
    tf = flops / (ms * 1e-3) / 1e12
    cs = clocks.summary()
    mhz = cs.get("sm_mhz") or 2070.0
    peak = 152 * 128 * 2 * mhz * 1e6 / 1e12
    print(json.dumps({
        "metric": "GDN forward with tree state routing, FP32 TFLOP/s on 1 GB300",
        "value": tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "tokens": N, "qk_heads": hk, "v_heads": hv, "head_dim": 128,
                   "l2": "inputs larger than L2, and L2 flushed between steps"},
        "tokens_per_s": N / (ms * 1e-3),
        "roofline": {"bound": "alu", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                     "peak_source": "152 SMs x 128 FP32 lanes x 2 flops x sampled SM clock", "traffic": None},
        "clocks": cs, "gpu_launches": args.steps * plan.info["gdn_levels"],
    }))


def partition_arm(args):
    """--op partition: the host partition planner (§3.3) on the workload at a
    token cap; no GPU. Reports the partitions, their lower bound and the peak
    tokens along a chain of partitions, with the planner's time."""
    import treegen
    import tree_packed_attention_gb300 as tpa

    w = treegen.workload(args.workload)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N = plan.num_tokens
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        r = tpa.tree_partition(plan, args.cap)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    tries = int(plan.info["num_tries"])
    print(json.dumps({
        "metric": "node-boundary partitions under a token cap (host planner)", "value": r["num_parts"],
        "unit": "partitions", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": False, "vs_baseline": None, "data": "synthetic",
        "config": {"workload": w.name, "tokens": N, "cap_tokens": args.cap, "tries": tries},
        "lower_bound": max(-(-N // args.cap), tries), "peak_path_tokens": r["peak_path_tokens"],
        "largest_partition": int(r["tokens"].max()) if r["num_parts"] else 0,
        "planner_ms": 1e3 * statistics.median(times),
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra-workloads", default="3,4",
                    help="comma-separated workloads also timed and reported under 'workloads' "
                         "('' for none)")
    ap.add_argument("--op", default="attention", choices=["attention", "rope", "conv", "ce", "gdn", "partition",
                                                         "gateway"],
                    help="attention (the default and the headline), rope (tree RoPE on q and k), "
                         "conv (the tree-correct causal conv), ce (the fused weighted cross-entropy; "
                         "workload 6 unless --workload is given), gdn (GDN with tree state routing), "
                         "gateway (partition-gateway attention over the pieces of a --cap cut; "
                         "workload 4 unless --workload is given), "
                         "or partition (the host planner, no GPU)")
    ap.add_argument("--gdn-heads", type=int, default=16, help="query/key heads for --op gdn (value heads: 2x)")
    ap.add_argument("--vocab", type=int, default=151936, help="vocabulary for --op ce")
    ap.add_argument("--channels", type=int, default=4096, help="channels for --op conv")
    ap.add_argument("--cap", type=int, default=16384, help="token cap for --op partition")
    args = ap.parse_args()
    if args.op == "rope":
        rope_arm(args)
    elif args.op == "conv":
        conv_arm(args)
    elif args.op == "gdn":
        gdn_arm(args)
    elif args.op == "ce":
        if "--workload" not in sys.argv:
            args.workload = 6
        ce_arm(args)
    elif args.op == "partition":
        partition_arm(args)
    elif args.op == "gateway":
        if "--workload" not in sys.argv:
            args.workload = 4
        gateway_arm(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
