#!/usr/bin/env python3
"""Benchmark of paged-KV varlen attention on GB300: one JSON line on stdout.

A step is one pattn_forward call over one batch: the device plan, the fused
attention kernel (page gather, QK^T, mask, online softmax, PV, epilogue) and
the split-KV combine. The headline workload is the pure decode batch (64
sequences x 1 query token, KV lengths uniform in [1024, 8192], 32 query / 8
KV heads, head dim 128, pages of 64 shuffled over the pool); its metric is
KV GB/s (live K and V rows once per KV head, plus Q and O). The causal
prefill batch (4 x 8192 tokens, same heads) is reported alongside as
attention TFLOP/s. Inputs are seeded synthetic data (numpy PCG64, bf16).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) each rank runs its own batch of the same shape (weak
scaling, no collective on the data path); value = all ranks' bytes / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DECODE = 2   # workload numbers of workloads.named
# the headline metric, the same string on both arms (ours and the oracle's)
HEADLINE_METRIC = "decode KV GB/s (live K/V bytes once per KV head + Q + O, per second)"
PREFILL = 3
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the sources each profiled kernel is compiled from (its ncu summary names their hash)
KERNEL_SOURCES = {"decode": ["decode.cu", "merge.cuh", "ptx.cuh", "kernels.cuh"],
                  "prefill": ["attn.cu", "merge.cuh", "ptx.cuh", "kernels.cuh"]}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--prefill-steps", type=int, default=30)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["decode", "prefill"], default=None,
                    help="profiling runs: time one workload only")
    ap.add_argument("--workload", default=None,
                    help="time named workload(s) 1-5 (comma list or 'all'): one JSON line each")
    ap.add_argument("--fp8qk", action="store_true",
                    help="with --workload: the quantised-QK variant (pattn_forward_fp8qk)")
    ap.add_argument("--fp8", action="store_true",
                    help="with --workload: the fp8 Q/K/P/V variant (pattn_forward_fp8)")
    ap.add_argument("--workload-steps", type=int, default=0,
                    help="with --workload: time at most this many steps (profiling runs)")
    ap.add_argument("--append", action="store_true",
                    help="with --workload: each step first writes the query tokens' K/V rows into "
                         "their cache slots (pattn_forward_append)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


def kernel_source_hash(kind: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "paged_kv_flashattention_varlen_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kind: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"{kind}_attention_kernel_traffic.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    val = re.search(r"traffic_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not src or not val or src.group(1) != kernel_source_hash(kind):
        return None
    return float(val.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int):
        import torch
        self.proc = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={uuid}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------- our arm
def profiled_pass(pk, step, steps):
    """Per-kernel device times: a second pass with the library's launch events on
    (the events add a little time per call, so the headline pass runs without)."""
    import torch
    torch.cuda.synchronize()
    pk.profile_read()
    pk.profile_enable(True)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    pk.profile_enable(False)
    return pk.profile_read()


def step_stats(step, steps):
    """Distribution of single-step device times (ms): a separate pass with a CUDA
    event pair around every step on the launching stream."""
    import numpy as np
    import torch
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    t = np.array([a.elapsed_time(b) for a, b in ev])
    q = np.percentile(t, [50, 90, 95, 99])
    return {"count": int(steps), "mean": round(float(t.mean()), 5), "p50": round(float(q[0]), 5),
            "p90": round(float(q[1]), 5), "p95": round(float(q[2]), 5), "p99": round(float(q[3]), 5),
            "min": round(float(t.min()), 5), "max": round(float(t.max()), 5)}


def profiled_kernels(pk, step, steps):
    """As :func:`profiled_pass`, split by kernel: ((plan, cache write, decode,
    prefill, after) ms summed over the calls, calls)."""
    import torch
    torch.cuda.synchronize()
    pk.profile_read()
    pk.profile_enable(True)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    pk.profile_enable(False)
    return pk.profile_read_kernels()


def headline_config(workloads, wl, world: int) -> dict:
    """The headline workload's description, the same on both arms."""
    return {"workload": workloads.NAMES[DECODE - 1], "batch": wl.num_seqs, "q_per_seq": 1,
            "kv_len": "uniform [1024, 8192], seeded", "n_heads_q": wl.n_heads_q,
            "n_heads_kv": wl.n_heads_kv, "head_dim": wl.head_dim, "page_size": wl.page_size,
            "causal": wl.causal, "kv_bytes_per_step": wl.kv_bytes(),
            "l2": "inputs larger than L2 (KV pool %.2f GB > 129 MB)" % (wl.kv_pool.numel() * 2 / 1e9),
            "parallelism": f"weak x{world}: one batch per GPU, no collective"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import paged_kv_flashattention_varlen_gb300 as pk
    from paged_kv_flashattention_varlen_gb300 import build as pkbuild
    from paged_kv_flashattention_varlen_gb300 import dist as pdist
    import workloads

    rank, world, local = pdist.rank_world()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(pk.library_path()):
        pkbuild.build()
    pdist.barrier(dev)
    pk._lib.load()
    pk_peaks, peak_kind = peaks()
    if args.only == "prefill":
        res = run_prefill(args, pk, workloads, dev, world, pk_peaks, peak_kind)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return

    # ---- decode batch (headline)
    wl = workloads.named(DECODE) if rank == 0 else _reseeded(workloads, DECODE, rank)
    q, kv = wl.q.to(dev), wl.kv_pool.to(dev)
    bt, sl, cu = wl.block_table.to(dev), wl.seq_lens.to(dev), wl.cu_q.to(dev)
    out = torch.empty_like(q)

    def step():
        pk.forward(out, q, kv, bt, sl, cu, max_q=wl.max_q, max_kv=wl.max_kv,
                   n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                   num_pages=wl.num_pages, check=False)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if pk.device_status() != 0:
        raise RuntimeError("device error during warm-up")
    pdist.barrier(dev)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    pdist.barrier(dev)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    ms_max = pdist.max_over_ranks(ms, dev if world > 1 else None)
    t_plan, t_attn, t_comb, calls = profiled_pass(pk, step, min(args.steps, 500))
    stats = step_stats(step, min(args.steps, 500))
    status = pk.device_status()
    step_bytes = wl.kv_bytes() + wl.qo_bytes()
    ms_step = ms_max / args.steps
    value = world * step_bytes * args.steps / (ms_max * 1e-3) / 1e9
    attn_ms = t_attn / max(calls, 1)
    achieved = step_bytes / (attn_ms * 1e-3) / 1e9
    hbm = float(pk_peaks["hbm_gbs"])
    traffic = ncu_traffic("decode")
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic,
                "peak_source": f"{peak_kind} hbm_gbs", "nominal_frac": round(achieved / NOMINAL_HBM_GBS, 4),
                "kernel": "decode_kernel<128> (swap-AB)", "kernel_ms": round(attn_ms, 5),
                "share": {"plan": round(t_plan / max(t_plan + t_attn + t_comb, 1e-9), 4),
                          "attention": round(t_attn / max(t_plan + t_attn + t_comb, 1e-9), 4),
                          "combine": round(t_comb / max(t_plan + t_attn + t_comb, 1e-9), 4)},
                "algorithmic_bytes_per_launch": step_bytes}

    # ---- end to end through the host-buffer entry point (pinned memory)
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, pk, wl, dev, world, step_bytes)

    # ---- causal prefill (secondary)
    prefill = None if args.only == "decode" else run_prefill(args, pk, workloads, dev, world,
                                                              pk_peaks, peak_kind)

    line = {
        "metric": HEADLINE_METRIC,
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(workloads, wl, world),
        "roofline": roofline, "step_ms_stats": stats, "e2e": e2e, "gpu_launches": int(2 * args.steps),
        "clocks": clocks,
        "device_status": status, "prefill": prefill,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(args, pk, wl, dev, world, step_bytes):
    import torch
    from paged_kv_flashattention_varlen_gb300 import dist as pdist
    hq, hkv_, hbt = wl.q.pin_memory(), wl.kv_pool.pin_memory(), wl.block_table.pin_memory()
    hsl, hcu = wl.seq_lens.pin_memory(), wl.cu_q.pin_memory()
    hout = torch.empty_like(wl.q).pin_memory()

    def e2e_step():
        pk.forward_host(hout, hq, hkv_, hbt, hsl, hcu, max_q=wl.max_q, max_kv=wl.max_kv,
                        n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                        num_pages=wl.num_pages)

    e2e_step()
    pdist.barrier(dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_s = pdist.max_over_ranks(e0.elapsed_time(e1) * 1e-3, dev if world > 1 else None)
    h2d = (hq.numel() * 2 + hkv_.numel() * 2 + hbt.numel() * 4 + hsl.numel() * 4 + hcu.numel() * 4)
    e2e = {"value": round(world * step_bytes * args.e2e_steps / e2e_s / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(hout.numel() * 2),
           "ms_per_step": round(e2e_s * 1e3 / args.e2e_steps, 3),
           "api": "pattn_forward_host (pinned host buffers, copies inside the timed region)"}
    return e2e



def _reseeded(workloads, index, rank):
    import numpy as np
    # same shape, other values: another rank's batch
    base = workloads.named(index)
    lens = base.seq_lens.numpy()
    qls = base.q_lens()
    return workloads.make_paged(base.name, workloads.seed_for(index) + 7919 * rank, qls.tolist(),
                                lens.tolist(), base.n_heads_q, base.n_heads_kv, base.head_dim,
                                base.page_size, scale=base.scale, causal=base.causal,
                                extra_pages=base.num_pages - int(np.sum(-(-lens // 64))))


def run_prefill(args, pk, workloads, dev, world, pk_peaks, peak_kind):
    import torch
    from paged_kv_flashattention_varlen_gb300 import dist as pdist
    wl = workloads.named(PREFILL)
    q, kv = wl.q.to(dev), wl.kv_pool.to(dev)
    bt, sl, cu = wl.block_table.to(dev), wl.seq_lens.to(dev), wl.cu_q.to(dev)
    out = torch.empty_like(q)

    def step():
        pk.forward(out, q, kv, bt, sl, cu, max_q=wl.max_q, max_kv=wl.max_kv,
                   n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                   num_pages=wl.num_pages, check=False)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    pdist.barrier(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.prefill_steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = pdist.max_over_ranks(e0.elapsed_time(e1), dev if world > 1 else None)
    t_plan, t_attn, t_comb, calls = profiled_pass(pk, step, args.prefill_steps)
    stats = step_stats(step, args.prefill_steps)
    flops = 4.0 * wl.head_dim * wl.n_heads_q * wl.visible_pairs()
    attn_ms = t_attn / max(calls, 1)
    achieved = flops / (attn_ms * 1e-3) / 1e12
    peak = float(pk_peaks["bf16_tflops"])
    return {
        "workload": workloads.NAMES[PREFILL - 1], "metric": "causal prefill attention TFLOP/s",
        "value": round(world * flops * args.prefill_steps / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "steps": args.prefill_steps, "ms_per_step": round(ms / args.prefill_steps, 4),
        "flops_per_step": flops,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": ncu_traffic("prefill"), "peak_source": f"{peak_kind} bf16_tflops (burst)",
                     "nominal_frac": round(achieved / NOMINAL_BF16_TFLOPS, 4),
                     "kernel": "attn_kernel<128,128>", "kernel_ms": round(attn_ms, 4)},
        "step_ms_stats": stats, "gpu_launches": int(3 * args.prefill_steps),
    }


# --------------------------------------------------------------------- oracle (CPU)
def cpu_baseline(wl, seconds: float):
    """The float64 oracle as it stands, on the host cores, over whole passes of
    the same decode batch, repeated until `seconds` have passed."""
    import oracle
    n_threads = oracle.threads()
    bytes_per_pass = wl.kv_bytes() + wl.qo_bytes()
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.forward_workload(wl, n_threads=n_threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 1000:
            break
    return {"value": round(bytes_per_pass * reps / el / 1e9, 4), "unit": "GB/s", "cores": n_threads,
            "kind": "oracle",
            "sample": f"{reps} full pass(es) of the 64-sequence decode batch in {el:.1f} s "
                      f"(float64 C, {n_threads} threads)"}


def run_reference(args):
    """Reference arm: the float64 oracle on the host cores, same workload and metric."""
    from paged_kv_flashattention_varlen_gb300 import dist as pdist
    rank, world, _ = pdist.rank_world()
    if rank != 0:
        return
    import oracle
    import workloads
    oracle.build()
    wl = workloads.named(DECODE)
    n_threads = oracle.threads()
    bytes_per_pass = wl.kv_bytes() + wl.qo_bytes()
    # each step: a bounded sample of the batch (every sequence, a slice of the query rows)
    rows = list(range(wl.total_q))
    for _ in range(max(args.warmup, 0)):
        oracle.forward_workload(wl, rows=rows, n_threads=n_threads)
    steps = max(1, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.forward_workload(wl, rows=rows, n_threads=n_threads)
    el = time.perf_counter() - t0
    value = bytes_per_pass * steps / el / 1e9
    line = {
        "impl": "reference", "metric": HEADLINE_METRIC,
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": max(args.warmup, 0), "ms_per_step": round(el * 1e3 / steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": headline_config(workloads, wl, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n_threads, "kind": "oracle",
                         "sample": f"{steps} full pass(es) of the decode batch"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_workloads(args):
    """One JSON line per named workload: step time, KV GB/s, attention TFLOP/s and the
    attention kernels' fractions of the HBM and bf16 rooflines."""
    import torch

    import paged_kv_flashattention_varlen_gb300 as pk
    from paged_kv_flashattention_varlen_gb300 import build as pkbuild
    import workloads

    pkbuild.build()
    pk_peaks, peak_kind = peaks()
    hbm, tc = float(pk_peaks["hbm_gbs"]), float(pk_peaks["bf16_tflops"])
    idxs = [1, 2, 3, 4, 5] if args.workload == "all" else [int(x) for x in args.workload.split(",")]
    dev = torch.device("cuda", 0)
    for i in idxs:
        wl = workloads.named(i)
        q, kv = wl.q.to(dev), wl.kv_pool.to(dev)
        bt = None if wl.block_table is None else wl.block_table.to(dev)
        sl, cu = wl.seq_lens.to(dev), wl.cu_q.to(dev)
        out = torch.empty_like(q)
        k_new = v_new = None
        if args.append:
            k_new, v_new = (t.to(dev) for t in workloads.new_kv_rows(wl, 900 + i))

        def step():
            if args.fp8:
                pk.forward_fp8(out, q, kv, bt, sl, cu, max_q=wl.max_q, max_kv=wl.max_kv,
                               n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                               num_pages=wl.num_pages, check=False)
            elif args.fp8qk:
                pk.forward_fp8qk(out, q, kv, bt, sl, cu, max_q=wl.max_q, max_kv=wl.max_kv,
                                 n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                                 num_pages=wl.num_pages, check=False)
            elif args.append:
                pk.forward_append(out, q, k_new, v_new, kv, bt, sl, cu, max_q=wl.max_q,
                                  max_kv=wl.max_kv, n_heads_kv=wl.n_heads_kv, scale=wl.scale,
                                  causal=wl.causal, num_pages=wl.num_pages, check=False)
            else:
                pk.forward(out, q, kv, bt, sl, cu, max_q=wl.max_q, max_kv=wl.max_kv,
                           n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                           num_pages=wl.num_pages, check=False)

        flops = 4.0 * wl.head_dim * wl.n_heads_q * wl.visible_pairs()
        nbytes = wl.kv_bytes() + wl.qo_bytes()
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        est = 1e-3 * max(flops / 9e14, nbytes / 6e12, 2e-5) * 1e3
        steps = max(5, min(2000, int(1.0 / max(est, 1e-6))))
        if args.workload_steps > 0:
            steps = min(steps, args.workload_steps)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        kt, calls = profiled_kernels(pk, step, min(steps, 500))
        t_plan, t_write, t_attn, t_comb = kt[0], kt[1], kt[2] + kt[3], kt[4]
        ms = e0.elapsed_time(e1) / steps
        attn_ms = t_attn / max(calls, 1)
        line = {
            "workload": workloads.NAMES[i - 1], "steps": steps, "ms_per_step": round(ms, 5),
            "kv_gbs_step": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "tflops_step": round(flops / (ms * 1e-3) / 1e12, 1),
            "attention_kernels_ms": round(attn_ms, 5),
            "hbm_frac_attention": round(nbytes / (attn_ms * 1e-3) / 1e9 / hbm, 4),
            "tensor_frac_attention": round(flops / (attn_ms * 1e-3) / 1e12 / tc, 4),
            "plan_ms": round(t_plan / max(calls, 1), 5), "combine_ms": round(t_comb / max(calls, 1), 5),
            "decode_kernel_ms": round(kt[2] / max(calls, 1), 5),
            "prefill_kernel_ms": round(kt[3] / max(calls, 1), 5),
            "bytes": nbytes, "flops": flops, "peaks": f"{peak_kind}: hbm {hbm} GB/s, bf16 {tc} TFLOP/s",
            "device_status": pk.device_status(),
        }
        if args.fp8qk:
            # QK on e4m3 tensor cores (twice the bf16 rate), PV in bf16: the tensor
            # roofline time is 0.75 of the bf16 one; the quantisation passes are
            # the "cache write" slot of the per-kernel record
            line["workload"] += "+fp8qk"
            line["quant_ms"] = round(t_write / max(calls, 1), 5)
            line["tensor_frac_attention_fp8qk_roofline"] = round(
                flops / (attn_ms * 1e-3) / 1e12 / (tc / 0.75), 4)
        if args.fp8:
            # QK and PV on e4m3 tensor cores: half the bf16 roofline time
            line["workload"] += "+fp8"
            line["quant_ms"] = round(t_write / max(calls, 1), 5)
            line["tensor_frac_attention_fp8_roofline"] = round(
                flops / (attn_ms * 1e-3) / 1e12 / (2 * tc), 4)
        if args.append:
            # K and V rows of every query token read once and written once
            wbytes = 4 * int(wl.q.shape[0]) * wl.n_heads_kv * wl.head_dim * 2
            write_ms = t_write / max(calls, 1)
            line["workload"] += "+kv_write"
            line["kv_write_ms"] = round(write_ms, 5)
            line["kv_write_bytes"] = wbytes
            line["kv_write_hbm_frac"] = round(wbytes / (write_ms * 1e-3) / 1e9 / hbm, 4)
        print(json.dumps(line), flush=True)
        del q, kv, bt, sl, cu, out
        torch.cuda.empty_cache()


def main():
    args = parse()
    if args.workload:
        run_workloads(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
