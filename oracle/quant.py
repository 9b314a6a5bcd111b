"""Oracle of the quantised-QK variant (test infrastructure only): the
SageAttention2-style preparation phases of the GB10 "sage2" benchmark page
(phases ``k_mean_and_smoothing_preparation``, ``q_int8_quantization``,
``k_int8_subtract_mean_quantization``), with fp8 e4m3 codes in place of int8,
and the attention over the dequantised Q and K.

Readings (the page names the phases and gives the scheduler's block sizes
``warp_q`` 32 and ``cta_k`` = ``warp_k`` 64, nothing else):

* smoothing: per (sequence, KV head, channel) the mean of K over the
  sequence's keys is subtracted. Every score of a query row then moves by the
  same q . mean, which the softmax cancels (exact in real arithmetic).
* K codes: one scale per (64-key block of a sequence, KV head) -- the page's
  64-key K block; for a paged cache that is one page.
* Q codes: one scale per query row (token, head), finer than the 32-row warp
  block, so that no block crosses a sequence boundary.
* scale = amax / 448 in fp32 (448 = largest e4m3 value; amax = 0 gives scale 1
  and all-zero codes); code = e4m3 round-to-nearest-even of (x / scale)
  computed in fp32 and saturated to +-448.
* the mean is the exact sum of the bf16 keys (exact in float64) divided by L in
  float64, then rounded to fp32; x = key - mean in fp32.

Both sides take every rounding decision in the same precision, so the codes
and scales are reproducible bit for bit.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_codes(x32: np.ndarray) -> np.ndarray:
    """fp32 -> e4m3 bytes (round to nearest even, saturated to +-448)."""
    import torch
    x = np.clip(np.asarray(x32, dtype=np.float32), -E4M3_MAX, E4M3_MAX)
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    """e4m3 bytes -> float64 values."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _scale(amax32: np.ndarray) -> np.ndarray:
    a = np.asarray(amax32, dtype=np.float32)
    s = (a / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(a > 0, s, np.float32(1.0)).astype(np.float32)


def _bf16_to_f32(t) -> np.ndarray:
    return t.detach().cpu().float().numpy().astype(np.float32)


def logical_k(kv_pool, block_table, seq_lens, b: int, page_size: int = 64, start: int = 0):
    """K of sequence b as fp32 [L, Hkv, D] (exact bf16 values)."""
    L = int(seq_lens[b])
    if block_table is None:
        return _bf16_to_f32(kv_pool[0, start:start + L])
    j = np.arange(L)
    bt = np.asarray(block_table[b].cpu().numpy() if hasattr(block_table, "cpu") else block_table[b])
    pages = bt[j // page_size]
    pool = kv_pool.detach().cpu()
    return pool[pages, 0, j % page_size].float().numpy().astype(np.float32)


def k_mean(k32: np.ndarray) -> np.ndarray:
    """Per (KV head, channel) mean over the keys: exact float64 sum / L, rounded to fp32."""
    L = k32.shape[0]
    if L == 0:
        return np.zeros(k32.shape[1:], dtype=np.float32)
    return (k32.astype(np.float64).sum(axis=0) / L).astype(np.float32)


def quantize_k(k32: np.ndarray, mean32: np.ndarray, block: int = 64):
    """Smoothed K -> (codes uint8 [nblk*block, Hkv, D], scales fp32 [nblk, Hkv]).
    Rows past L of the last block are zero codes."""
    L, H, D = k32.shape
    nblk = (L + block - 1) // block
    x = (k32 - mean32[None]).astype(np.float32)
    codes = np.zeros((nblk * block, H, D), dtype=np.uint8)
    scales = np.zeros((nblk, H), dtype=np.float32)
    for i in range(nblk):
        xb = x[i * block:(i + 1) * block]
        s = _scale(np.abs(xb).max(axis=(0, 2)))
        scales[i] = s
        codes[i * block:i * block + xb.shape[0]] = e4m3_codes((xb / s[None, :, None]).astype(np.float32))
    return codes, scales


def quantize_q(q32: np.ndarray):
    """Q fp32 [T, Hq, D] -> (codes uint8 [T, Hq, D], scales fp32 [T, Hq]), one scale per row."""
    s = _scale(np.abs(q32).max(axis=2))
    codes = e4m3_codes((q32 / s[:, :, None]).astype(np.float32))
    return codes, s


def quantize_workload(wl):
    """The codes and scales of a workload: dict with q_codes [T, Hq, D], q_scale [T, Hq],
    k_mean [B, Hkv, D], and per sequence b: k_codes[b] [nblk*64, Hkv, D], k_scale[b] [nblk, Hkv]."""
    q32 = _bf16_to_f32(wl.q)
    qc, qs = quantize_q(q32)
    means, kcs, kss = [], [], []
    start = 0
    for b in range(wl.num_seqs):
        k32 = logical_k(wl.kv_pool, wl.block_table, wl.seq_lens, b, wl.page_size, start)
        m = k_mean(k32)
        kc, ks = quantize_k(k32, m)
        means.append(m)
        kcs.append(kc)
        kss.append(ks)
        start += int(wl.seq_lens[b])
    return dict(q_codes=qc, q_scale=qs, k_mean=np.stack(means) if means else None, k_codes=kcs,
                k_scale=kss)


def attention_dequantized(wl, rows=None, qz=None):
    """float64 attention of the quantised-QK method: softmax(scale * q^ . k^) v
    with q^, k^ the dequantised (smoothed) Q and K and v the bf16 V, per query
    token (all, or the global token indices in ``rows``). Returns [n, Hq, D].

    Q rows are quantised independently, so only the requested ones are; K is
    quantised (and dequantised head by head) for the sequences those rows
    belong to. ``qz`` (from :func:`quantize_workload`) may be given instead.
    """
    cu = wl.cu_q.numpy().astype(np.int64)
    sl = wl.seq_lens.numpy().astype(np.int64)
    starts = np.concatenate([[0], np.cumsum(sl)])
    toks = np.arange(int(cu[-1])) if rows is None else np.asarray(list(rows), dtype=np.int64)
    G = wl.n_heads_q // wl.n_heads_kv
    if qz is None:
        qc, qs = quantize_q(_bf16_to_f32(wl.q[torch_index(toks)]))
    else:
        qc, qs = qz["q_codes"][toks], qz["q_scale"][toks]
    q_deq = e4m3_values(qc) * qs.astype(np.float64)[:, :, None]
    seq_of = np.searchsorted(cu, toks, side="right") - 1
    pool = wl.kv_pool.detach().cpu()
    out = np.zeros((len(toks), wl.n_heads_q, wl.head_dim), dtype=np.float64)
    for b in np.unique(seq_of):
        b = int(b)
        L = int(sl[b])
        ql = int(cu[b + 1] - cu[b])
        if qz is None:
            k32 = logical_k(wl.kv_pool, wl.block_table, wl.seq_lens, b, wl.page_size, int(starts[b]))
            kc, ks = quantize_k(k32, k_mean(k32))
        else:
            kc, ks = qz["k_codes"][b], qz["k_scale"][b]
        if wl.block_table is None:
            v = pool[1, starts[b]:starts[b] + L]
        else:
            j = np.arange(L)
            v = pool[wl.block_table[b].numpy()[j // wl.page_size], 1, j % wl.page_size]
        mine = np.nonzero(seq_of == b)[0]
        for hk in range(wl.n_heads_kv):
            k = e4m3_values(kc[:L, hk]) * np.repeat(ks[:, hk].astype(np.float64), 64)[:L, None]
            vh = v[:, hk].double().numpy()
            for n in mine:
                pos = L - ql + (int(toks[n]) - int(cu[b]))
                nk = min(L, pos + 1) if wl.causal else L
                if nk <= 0:
                    continue
                for h in range(hk * G, (hk + 1) * G):
                    s = (k[:nk] @ q_deq[n, h]) * wl.scale
                    w = np.exp(s - s.max())
                    out[n, h] = (w @ vh[:nk]) / w.sum()
    return out


def torch_index(idx):
    import torch
    return torch.as_tensor(np.asarray(idx, dtype=np.int64))
