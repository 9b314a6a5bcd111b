#!/usr/bin/env python3
"""Benchmark of paged-KV varlen attention on GB300: one JSON line on stdout.

A step is one pattn_forward call over one batch: the device plan and the
attention kernels (page gather, QK^T, mask, online softmax, PV, epilogue, and
the in-kernel merge of split-KV partials). Inputs are seeded synthetic data
(numpy PCG64, bf16), resident in HBM before any timed region.

Headline: the pure decode batch (64 sequences x 1 query token, KV lengths
uniform in [1024, 8192], 32 query / 8 KV heads, head dim 128, pages of 64
shuffled over the pool), metric KV GB/s (live K and V rows once per KV head,
plus Q and O). `value` and `ms_per_step` time exactly `--steps` steps between
one CUDA event pair.

Every named workload (the tiny paged decode, the decode batch, the causal
4 x 8192 prefill, the non-causal 37,810-token batch and the mixed batch) then
gets one interleaved timing pass (`measure`) under its own clock record: plain
steps (each in its own event pair, for the step-time distribution) alternate
with steps that carry the library's per-launch events, so the attention-kernel
times and the step times of an entry come from the same pass and clocks. The
line's `roofline` is the decode kernel's, from that pass on the headline batch;
`workloads` holds all five entries, each with its roofline (HBM, tensor, or
both for the mixed batch) and the float64 oracle's time on the host cores.

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
                  "prefill": ["attn.cu", "prefill.cuh", "merge.cuh", "ptx.cuh", "kernels.cuh"],
                  "prefill_two_q": ["attn2q.cu", "prefill.cuh", "merge.cuh", "ptx.cuh", "kernels.cuh"]}
# the kernel each named workload's roofline traffic is taken for (its ncu summary)
TRAFFIC_KIND = {2: "decode", 3: "prefill", 4: "prefill_two_q"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--prefill-steps", type=int, default=0,
                    help="cap on the steps of each named workload's interleaved pass (0: by --workload-seconds)")
    ap.add_argument("--workload-seconds", type=float, default=1.0,
                    help="seconds of the interleaved timing pass of each named workload")
    ap.add_argument("--no-workloads", action="store_true",
                    help="headline only: skip the other named workloads")
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
    ap.add_argument("--scale-down", type=int, default=1,
                    help="with --workload: divide the token counts by this (smaller cases for profiling)")
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
def _events(n):
    import torch
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]


def _stats(t):
    import numpy as np
    t = np.asarray(t, dtype=np.float64)
    q = np.percentile(t, [50, 90, 95, 99])
    return {"count": int(t.size), "mean": round(float(t.mean()), 5), "p50": round(float(q[0]), 5),
            "p90": round(float(q[1]), 5), "p95": round(float(q[2]), 5), "p99": round(float(q[3]), 5),
            "min": round(float(t.min()), 5), "max": round(float(t.max()), 5)}


def measure(pk, step, seconds, device_index, flush=None, max_steps=0):
    """One interleaved timing pass of a workload, under one clock record.

    Blocks of plain steps and blocks of profiled steps alternate (the library's
    per-launch CUDA events on in the latter; those events turn the dependent-
    launch overlap off, so they are kept out of the plain steps). Every step
    has its own CUDA event pair on the launching stream; `flush` (a write of
    twice the L2 size) runs before each step, outside the pair. Returns the
    plain steps' time distribution, the profiled steps' mean and the per-kernel
    device times of the profiled steps, all from the same pass, so that each
    kernel time is part of a step timed under the same clocks."""
    import torch
    for _ in range(3):
        if flush:
            flush()
        step()
    torch.cuda.synchronize()
    (a, b), = _events(1)
    if flush:
        flush()
    a.record()
    step()
    b.record()
    torch.cuda.synchronize()
    est_ms = max(a.elapsed_time(b), 1e-3)
    total = max(4, int(seconds * 1e3 / est_ms))
    if max_steps > 0:
        total = max(2, min(total, max_steps))
    total = min(total, 8000)  # the library keeps at most 4096 profiled calls
    half = max(1, min(500, int(50.0 / est_ms), total // 2))
    blocks = max(1, total // (2 * half))
    pk.profile_read()
    sampler = ClockSampler(device_index)
    time.sleep(0.25)
    plain, prof = [], []
    for _ in range(blocks):
        for profiled in (False, True):
            evs = _events(half)
            pk.profile_enable(profiled)
            for x, y in evs:
                if flush:
                    flush()
                x.record()
                step()
                y.record()
            pk.profile_enable(False)
            torch.cuda.synchronize()
            (prof if profiled else plain).extend(x.elapsed_time(y) for x, y in evs)
    clocks = sampler.stop()
    kt, calls = pk.profile_read_kernels()
    n = max(calls, 1)
    kernel_ms = {"plan": kt[0] / n, "cache_write_or_quant": kt[1] / n, "decode": kt[2] / n,
                 "prefill": kt[3] / n, "after": kt[4] / n}
    return {"plain": plain, "profiled_ms_per_step": sum(prof) / max(len(prof), 1),
            "kernel_ms": kernel_ms, "calls": calls, "clocks": clocks}


def launches_per_step(wl) -> int:
    """Kernels pattn_forward launches for this batch: the plan, the decode kernel
    when some unit may hold at most 16 packed rows (the GQA group fits and the
    bounds leave room for a sequence of at most 16 / G queries: every sequence
    holds at least total_q - (B - 1) * max_q), the prefill kernel when some unit
    may hold more than 16 packed rows."""
    g = wl.n_heads_q // wl.n_heads_kv
    dec = g <= 16 and (wl.total_q - (wl.num_seqs - 1) * max(wl.max_q, 0)) * g <= 16
    pre = (not dec) or wl.max_q * g > 16
    return 1 + int(dec) + int(pre)


KERNEL_NAMES = {1: "attn_kernel<256,64> (head_dim 256, one CTA)",
                2: "decode_kernel<128> (swap-AB)",
                3: "attn_kernel<128,128> (one q tile per CTA)",
                4: "attn2q_kernel (head_dim 128, two q tiles per CTA)",
                5: "decode_kernel<256> then attn_kernel<256,128,pair> (cta_group::2)"}
L2_NOTES = {1: "cold L2: a %d MB buffer written before every step, outside its events",
            2: "inputs larger than L2 (KV pool %.2f GB > 129 MB)",
            3: "inputs larger than L2 (KV pool %.2f GB > 129 MB)",
            4: "inputs larger than L2 (K/V planes %.2f GB > 129 MB)",
            5: "inputs larger than L2 (KV pool %.2f GB > 129 MB)"}
L2_FLUSH_BYTES = 2 * 129 * 1000 * 1000


def workload_entry(idx, wl, meas, pk_peaks, peak_kind):
    """Step time, attention-kernel time and the roofline of SURVEY-style
    accounting for one named workload: HBM for the decode batches, tensor for
    the prefill batches, max(bytes / BW, FLOPs / peak) for the mixed batch."""
    flops = 4.0 * wl.head_dim * wl.n_heads_q * wl.visible_pairs()
    nbytes = wl.kv_bytes() + wl.qo_bytes()
    km = meas["kernel_ms"]
    t_attn = km["decode"] + km["prefill"]
    hbm = float(pk_peaks["hbm_gbs"])
    tc = float(pk_peaks["bf16_tflops"])
    tcs = float(pk_peaks.get("bf16_tflops_sustained", tc))
    st = _stats(meas["plain"])
    if idx in (1, 2):
        ach = nbytes / (t_attn * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "peak_source": f"{peak_kind} hbm_gbs",
                "nominal_frac": round(ach / NOMINAL_HBM_GBS, 4),
                "algorithmic_bytes_per_launch": nbytes}
    elif idx in (3, 4):
        ach = flops / (t_attn * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": tcs, "unit": "TFLOP/s",
                "frac": round(ach / tcs, 4),
                "peak_source": f"{peak_kind} bf16_tflops_sustained (the kernel loops for seconds)",
                "frac_of_burst_peak": round(ach / tc, 4), "burst_peak": tc,
                "nominal_frac": round(ach / NOMINAL_BF16_TFLOPS, 4), "algorithmic_flops_per_launch": flops}
    else:
        t_bw = nbytes / (hbm * 1e9) * 1e3
        t_tc = flops / (tcs * 1e12) * 1e3
        roof = {"bound": "hbm+tensor", "frac": round(max(t_bw, t_tc) / t_attn, 4),
                "hbm_component": {"achieved": round(nbytes / (t_attn * 1e-3) / 1e9, 1), "peak": hbm,
                                  "unit": "GB/s", "frac": round(t_bw / t_attn, 4), "roofline_ms": round(t_bw, 5)},
                "tensor_component": {"achieved": round(flops / (t_attn * 1e-3) / 1e12, 1), "peak": tcs,
                                     "unit": "TFLOP/s", "frac": round(t_tc / t_attn, 4),
                                     "roofline_ms": round(t_tc, 5)},
                "frac_of_burst_tensor_peak": round(max(t_bw, flops / (tc * 1e12) * 1e3) / t_attn, 4),
                "peak_source": f"{peak_kind} hbm_gbs and bf16_tflops_sustained",
                "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops}
    roof.update({"kernel": KERNEL_NAMES[idx], "kernel_ms": round(t_attn, 5),
                 "decode_kernel_ms": round(km["decode"], 5), "prefill_kernel_ms": round(km["prefill"], 5),
                 "plan_ms": round(km["plan"], 5), "profiled_ms_per_step": round(meas["profiled_ms_per_step"], 5),
                 "source": "kernel_ms, profiled_ms_per_step and ms_per_step come from one interleaved pass "
                           "(alternating plain and profiled blocks under one clock record)"})
    if idx == 1:
        l2 = L2_NOTES[1] % (L2_FLUSH_BYTES // 1000000)
    else:
        l2 = L2_NOTES[idx] % (wl.kv_pool.numel() * 2 / 1e9)
    return {"workload": wl.name, "ms_per_step": st["mean"], "step_ms_stats": st,
            "kv_gbs_step": round(nbytes / (st["mean"] * 1e-3) / 1e9, 1),
            "tflops_step": round(flops / (st["mean"] * 1e-3) / 1e12, 1),
            "roofline": roof, "clocks": meas["clocks"], "l2": l2,
            "gpu_launches_per_step": launches_per_step(wl)}


def headline_config(workloads, wl, world: int) -> dict:
    """The headline workload's description, the same on both arms."""
    return {"workload": workloads.NAMES[DECODE - 1], "batch": wl.num_seqs, "q_per_seq": 1,
            "kv_len": "uniform [1024, 8192], seeded", "n_heads_q": wl.n_heads_q,
            "n_heads_kv": wl.n_heads_kv, "head_dim": wl.head_dim, "page_size": wl.page_size,
            "causal": wl.causal, "kv_bytes_per_step": wl.kv_bytes(),
            "l2": "inputs larger than L2 (KV pool %.2f GB > 129 MB)" % (wl.kv_pool.numel() * 2 / 1e9),
            "parallelism": f"weak x{world}: one batch per GPU, no collective"}


def _device_inputs(wl, dev):
    bt = None if wl.block_table is None else wl.block_table.to(dev)
    return wl.q.to(dev), wl.kv_pool.to(dev), bt, wl.seq_lens.to(dev), wl.cu_q.to(dev)


def _forward_step(pk, wl, q, kv, bt, sl, cu, out):
    def step():
        pk.forward(out, q, kv, bt, sl, cu, max_q=wl.max_q, max_kv=wl.max_kv,
                   n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                   num_pages=wl.num_pages, check=False)
    return step


def run_named(pk, workloads, idx, dev, local, seconds, max_steps, pk_peaks, peak_kind, oracle_s):
    """Measure one named workload (and time the oracle on it when oracle_s > 0)."""
    import torch
    wl = workloads.named(idx)
    q, kv, bt, sl, cu = _device_inputs(wl, dev)
    out = torch.empty_like(q)
    flush = None
    if idx == 1:
        buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        flush = lambda: buf.fill_(1)  # noqa: E731
    meas = measure(pk, _forward_step(pk, wl, q, kv, bt, sl, cu, out), seconds, local, flush, max_steps)
    entry = workload_entry(idx, wl, meas, pk_peaks, peak_kind)
    entry["device_status"] = pk.device_status()
    if idx in TRAFFIC_KIND:
        entry["roofline"]["traffic"] = ncu_traffic(TRAFFIC_KIND[idx])
    del q, kv, bt, sl, cu, out
    torch.cuda.empty_cache()
    if oracle_s > 0:
        entry["oracle"] = oracle_time(idx, wl, entry["ms_per_step"])
    return entry


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
        res = run_named(pk, workloads, PREFILL, dev, local, args.workload_seconds, args.prefill_steps,
                        pk_peaks, peak_kind, 0)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return

    # ---- decode batch (headline): exactly `steps` steps between one event pair
    wl = workloads.named(DECODE) if rank == 0 else _reseeded(workloads, DECODE, rank)
    q, kv, bt, sl, cu = _device_inputs(wl, dev)
    out = torch.empty_like(q)
    step = _forward_step(pk, wl, q, kv, bt, sl, cu, out)
    # the clock sampler starts first (it needs a moment before the timed region);
    # the warm-up steps then run right before the timed ones, so that the timed
    # region does not begin on a GPU that has sat idle
    sampler = ClockSampler(local)
    time.sleep(0.3)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if pk.device_status() != 0:
        raise RuntimeError("device error during warm-up")
    pdist.barrier(dev)
    torch.cuda.synchronize()
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
    status = pk.device_status()
    step_bytes = wl.kv_bytes() + wl.qo_bytes()
    ms_step = ms_max / args.steps
    value = world * step_bytes * args.steps / (ms_max * 1e-3) / 1e9

    # ---- the decode kernel's roofline: an interleaved pass of the same batch
    meas = measure(pk, step, args.workload_seconds, local)
    head_entry = workload_entry(DECODE, wl, meas, pk_peaks, peak_kind)
    roofline = dict(head_entry["roofline"])
    roofline.update({"traffic": ncu_traffic("decode"), "pass_ms_per_step": head_entry["ms_per_step"],
                     "pass_clocks": meas["clocks"], "pass_steps": len(meas["plain"]) + meas["calls"]})

    # ---- end to end through the host-buffer entry point (pinned memory)
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, pk, wl, dev, world, step_bytes)
    del q, kv, bt, sl, cu, out
    torch.cuda.empty_cache()

    line = {
        "metric": HEADLINE_METRIC,
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(workloads, wl, world),
        "roofline": roofline, "step_ms_stats": head_entry["step_ms_stats"], "e2e": e2e,
        "gpu_launches": int(launches_per_step(wl) * args.steps),
        "clocks": clocks, "device_status": status,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
        head_entry["oracle"] = {"ms_per_step": round(line["cpu_baseline"]["ms_per_pass"], 3),
                                "kind": "oracle, full passes", "cores": line["cpu_baseline"]["cores"],
                                "gpu_speedup": round(line["cpu_baseline"]["ms_per_pass"] / head_entry["ms_per_step"], 1)}
    del wl

    # ---- the other named workloads (one GPU run only): same interleaved pass each
    if world == 1 and not args.no_workloads and args.only is None:
        entries = {}
        for idx in (1, 3, 4, 5):
            e = run_named(pk, workloads, idx, dev, local, args.workload_seconds, args.prefill_steps,
                          pk_peaks, peak_kind, 0 if args.no_cpu_baseline else 1)
            entries[workloads.NAMES[idx - 1]] = e
        entries[workloads.NAMES[DECODE - 1]] = head_entry
        line["workloads"] = {workloads.NAMES[i - 1]: entries[workloads.NAMES[i - 1]] for i in (1, 2, 3, 4, 5)}
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
                      f"(float64 C, {n_threads} threads)",
            "ms_per_pass": el * 1e3 / reps}


def _strided(first, end, n):
    """n rows spread evenly over [first, end): the oracle's cost per row grows
    along a causal sequence, so an even spread keeps the mean unbiased."""
    import numpy as np
    stride = max(1, (end - first) // max(n, 1))
    return list(range(first + stride // 2, end, stride))


def oracle_time(idx, wl, gpu_ms):
    """The float64 oracle as it stands on the host cores, on one named workload:
    whole passes of the tiny decode; the mixed batch's decode rows in full with
    its chunk rows sampled; 1024 (causal prefill) or 128 (non-causal) evenly
    spread query rows x all heads of the prefill batches. Sampled parts are
    extrapolated linearly per row (output rows are independent)."""
    import oracle
    n_threads = oracle.threads()
    total = wl.total_q

    def timed(rows):
        t0 = time.perf_counter()
        oracle.forward_workload(wl, rows=rows, n_threads=n_threads)
        return time.perf_counter() - t0

    if idx == 1:
        el = min(timed(None) for _ in range(5))
        ms, kind = el * 1e3, "full pass (best of 5)"
    elif idx == 5:
        qls = wl.q_lens()
        n_dec = int((qls == 1).sum())
        t_dec = timed(list(range(n_dec)))
        rows = _strided(n_dec, total, 512)
        t_chunk = timed(rows) * (total - n_dec) / len(rows)
        ms = (t_dec + t_chunk) * 1e3
        kind = (f"decode rows in full ({t_dec * 1e3:.1f} ms); chunk rows extrapolated from {len(rows)} "
                f"of {total - n_dec} evenly spread rows ({t_chunk * 1e3:.1f} ms)")
    else:
        n = 1024 if idx == 3 else 128
        rows = _strided(0, total, n)
        ms = timed(rows) * total / len(rows) * 1e3
        kind = f"extrapolated from {len(rows)} of {total} evenly spread query rows x all heads"
    return {"ms_per_step": round(ms, 3), "kind": kind, "cores": n_threads,
            "gpu_speedup": round(ms / gpu_ms, 1)}


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
        wl = workloads.named(i, scale_down=args.scale_down)
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
        meas = measure(pk, step, args.workload_seconds, 0, None, args.workload_steps)
        km = meas["kernel_ms"]
        t_write = km["cache_write_or_quant"]
        attn_ms = km["decode"] + km["prefill"]
        st = _stats(meas["plain"])
        ms = st["mean"]
        line = {
            "workload": workloads.NAMES[i - 1] + (f"/{args.scale_down}" if args.scale_down > 1 else ""),
            "steps": st["count"], "ms_per_step": round(ms, 5),
            "kv_gbs_step": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "tflops_step": round(flops / (ms * 1e-3) / 1e12, 1),
            "attention_kernels_ms": round(attn_ms, 5),
            "hbm_frac_attention": round(nbytes / (attn_ms * 1e-3) / 1e9 / hbm, 4),
            "tensor_frac_attention": round(flops / (attn_ms * 1e-3) / 1e12 / tc, 4),
            "plan_ms": round(km["plan"], 5), "combine_ms": round(km["after"], 5),
            "decode_kernel_ms": round(km["decode"], 5),
            "prefill_kernel_ms": round(km["prefill"], 5),
            "profiled_ms_per_step": round(meas["profiled_ms_per_step"], 5),
            "bytes": nbytes, "flops": flops, "peaks": f"{peak_kind}: hbm {hbm} GB/s, bf16 {tc} TFLOP/s",
            "clocks": meas["clocks"], "device_status": pk.device_status(),
        }
        if args.fp8qk:
            # QK on e4m3 tensor cores (twice the bf16 rate), PV in bf16: the tensor
            # roofline time is 0.75 of the bf16 one; the quantisation passes are
            # the quantisation slot of the per-kernel record
            line["workload"] += "+fp8qk"
            line["quant_ms"] = round(t_write, 5)
            line["tensor_frac_attention_fp8qk_roofline"] = round(
                flops / (attn_ms * 1e-3) / 1e12 / (tc / 0.75), 4)
        if args.fp8:
            # QK and PV on e4m3 tensor cores: half the bf16 roofline time
            line["workload"] += "+fp8"
            line["quant_ms"] = round(t_write, 5)
            line["tensor_frac_attention_fp8_roofline"] = round(
                flops / (attn_ms * 1e-3) / 1e12 / (2 * tc), 4)
        if args.append:
            # K and V rows of every query token read once and written once, by the
            # plan grid's extra CTAs while the plan is made (inside plan_ms)
            wbytes = 4 * int(wl.q.shape[0]) * wl.n_heads_kv * wl.head_dim * 2
            line["workload"] += "+kv_write"
            line["kv_write_bytes"] = wbytes
            line["kv_write"] = "in the plan grid (plan_ms includes it); no launch of its own"
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
