"""Shared helpers of the GPU parity tests: move a workload to the device, run the
library through its C ABI, compare with the float64 oracle."""
import numpy as np
import torch

import oracle

# Parity bar on the bf16 outputs against the float64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def to_device(wl):
    dev = torch.device("cuda:0")
    return dict(
        q=wl.q.to(dev), kv=wl.kv_pool.to(dev),
        bt=None if wl.block_table is None else wl.block_table.to(dev),
        sl=wl.seq_lens.to(dev), cu=wl.cu_q.to(dev),
    )


def run_gpu(wl, d=None, out=None, check=True):
    import paged_kv_flashattention_varlen_gb300 as pk
    d = d or to_device(wl)
    if out is None:
        out = torch.full_like(d["q"], float("nan"))
    pk.forward(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q, max_kv=wl.max_kv,
               n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
               num_pages=wl.num_pages, check=check)
    torch.cuda.synchronize()
    return out


def errors(gpu_rows, ref_rows):
    g = gpu_rows.float().cpu().numpy().astype(np.float64)
    diff = np.abs(g - ref_rows)
    return float(diff.max()) if diff.size else 0.0, float(diff.mean()) if diff.size else 0.0


def assert_parity(gpu_out, wl, rows=None, n_threads=0):
    ref, _ = oracle.forward_workload(wl, rows=rows, n_threads=n_threads)
    got = gpu_out if rows is None else gpu_out[torch.as_tensor(rows, device=gpu_out.device)]
    g = got.float().cpu().numpy()
    assert np.isfinite(g).all(), "non-finite output"
    mx, mean = errors(got, ref)
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"max |err| {mx:.3e}, mean |err| {mean:.3e}"
    return mx, mean


def sample_rows(wl, per_seq=6, tile=None, seed=0, every_boundary=False, min_rows=0):
    """Query tokens the oracle computes one by one: the first and last rows of
    every sequence, rows at q-tile boundaries (tile-1, tile, tile+1) and seeded
    random rows.

    With ``every_boundary`` every q-tile boundary of every sequence is taken
    (so every q tile, and with all heads every work item, has checked rows);
    otherwise three boundaries per sequence. Random rows (at least ``per_seq``
    per sequence) are added until there are ``min_rows`` rows in all."""
    rng = np.random.default_rng(seed)
    cu = wl.cu_q.numpy().astype(np.int64)
    G = wl.n_heads_q // wl.n_heads_kv
    T = tile or max(1, 128 // G)
    rows = set()
    live = []
    for b in range(wl.num_seqs):
        a, e = int(cu[b]), int(cu[b + 1])
        if e == a:
            continue
        live.append((a, e))
        rows.update({a, e - 1})
        ks = range(1, (e - a + T - 1) // T) if every_boundary else (1, (e - a) // (2 * T), (e - a) // T - 1)
        for k in ks:
            for off in (-1, 0, 1):
                t = a + k * T + off
                if a <= t < e:
                    rows.add(t)
        rows.update(int(x) for x in rng.integers(a, e, size=min(per_seq, e - a)))
    total = sum(e - a for a, e in live)
    while live and len(rows) < min(min_rows, total):
        a, e = live[int(rng.integers(0, len(live)))]
        rows.add(int(rng.integers(a, e)))
    return sorted(rows)
