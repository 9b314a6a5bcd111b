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
* scale = amax / 448 in fp32 (448 = largest e4m3 value); code = e4m3
  round-to-nearest-even of x * inv, the product rounded to fp32, with
  inv = 448 / amax in fp32 (capped at the largest finite fp32), saturated to
  +-448. amax = 0 gives scale 1 and all-zero codes. amax is taken as C's fmaxf
  does, ignoring NaN. The page fixes no precision for the division by the
  scale; one reciprocal per block and a multiply per element is the plain
  reading of "divide by the scale" on a GPU, and the dequantised value
  code * scale differs from x by the e4m3 rounding plus a few fp32 ulps.
* the mean is summed exactly in fixed point: each bf16 key value is clamped to
  +-1024 and rounded (to nearest even) to a multiple of 2^-32, the integer
  counts are added exactly, and mean = count * 2^-32 / L in float64, rounded
  to fp32; x = key - mean in fp32. This is the plain mean of K for keys of
  magnitude 2^-25 ... 1024 (every bf16 value there lies on the 2^-32 grid);
  any per-channel offset is a valid smoothing, since the softmax cancels it.

Both sides take every rounding decision in the same precision, so the codes
and scales are reproducible bit for bit.

Test infrastructure only: the product path never imports this module.
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


FLT_MAX = np.float32(np.finfo(np.float32).max)


def _amax(x32: np.ndarray, axis) -> np.ndarray:
    """max |x| over ``axis``, NaN ignored (0 for an all-NaN or all-zero block)."""
    return np.fmax.reduce(np.abs(np.asarray(x32, dtype=np.float32)), axis=axis, initial=np.float32(0))


def _scale(amax32: np.ndarray) -> np.ndarray:
    """Dequantisation scale amax / 448 in fp32 (1 where amax = 0)."""
    a = np.asarray(amax32, dtype=np.float32)
    with np.errstate(divide="ignore"):
        s = (a / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(a > 0, s, np.float32(1.0)).astype(np.float32)


def _inv_scale(amax32: np.ndarray) -> np.ndarray:
    """Quantisation multiplier 448 / amax in fp32, capped at the largest finite fp32 (1 where amax = 0)."""
    a = np.asarray(amax32, dtype=np.float32)
    with np.errstate(divide="ignore", over="ignore"):
        inv = np.minimum((np.float32(E4M3_MAX) / np.where(a > 0, a, np.float32(1))).astype(np.float32), FLT_MAX)
    return np.where(a > 0, inv, np.float32(1.0)).astype(np.float32)


def _codes(x32: np.ndarray, inv32: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore", over="ignore"):
        return e4m3_codes((np.asarray(x32, dtype=np.float32) * inv32).astype(np.float32))


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


SUM_CLAMP = 1024.0
SUM_UNIT = 2.0 ** 32


def k_sum_units(k32: np.ndarray) -> np.ndarray:
    """Per (KV head, channel) exact sum of the keys in units of 2^-32 (int64):
    each value clamped to +-1024 (NaN to the lower bound, as C's fmaxf does)
    and rounded to the nearest multiple of 2^-32, ties to even."""
    x = np.fmin(np.fmax(np.asarray(k32, dtype=np.float32), np.float32(-SUM_CLAMP)), np.float32(SUM_CLAMP))
    units = np.rint(x * np.float32(SUM_UNIT)).astype(np.int64)
    return units.sum(axis=0, dtype=np.int64)


def k_mean(k32: np.ndarray) -> np.ndarray:
    """Per (KV head, channel) smoothing offset: the fixed-point sum * 2^-32 / L in
    float64, rounded to fp32 (the mean of K for keys within the grid's range)."""
    L = k32.shape[0]
    if L == 0:
        return np.zeros(k32.shape[1:], dtype=np.float32)
    return (k_sum_units(k32).astype(np.float64) * (1.0 / SUM_UNIT) / L).astype(np.float32)


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
        amax = _amax(xb, axis=(0, 2))
        scales[i] = _scale(amax)
        codes[i * block:i * block + xb.shape[0]] = _codes(xb, _inv_scale(amax)[None, :, None])
    return codes, scales


def quantize_q(q32: np.ndarray):
    """Q fp32 [T, Hq, D] -> (codes uint8 [T, Hq, D], scales fp32 [T, Hq]), one scale per row."""
    amax = _amax(q32, axis=2)
    return _codes(q32, _inv_scale(amax)[:, :, None]), _scale(amax)


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


# ---------------------------------------------------------------------------
# fp8 P.V: the V phases of the same page (``v_fp8_transpose_scale_quantization``
# with its transpose/pad/permute and scale/fp8 parts, ``v_scale_fp8_quantization``)
# and the attention with e4m3 P and V.
#
# Readings: one V scale per (sequence, KV head, channel) over the sequence's keys
# (a per-channel scale is constant along the keys, so it factors out of P.V and
# is applied to O); the codes are stored transposed, keys innermost, in tiles of
# 128 keys padded with zero codes: [tile][KV head][channel][128 keys].

V_TILE = 128
P_SCALE_LOG2 = 2       # P is coded as e4m3 of p * 2^2
P_SLACK_LOG2 = 6       # codes stay at most 2^(2 + 6): the running max may trail by up to 2^6


def logical_v(kv_pool, block_table, seq_lens, b: int, page_size: int = 64, start: int = 0):
    """V of sequence b as fp32 [L, Hkv, D] (exact bf16 values)."""
    L = int(seq_lens[b])
    if block_table is None:
        return _bf16_to_f32(kv_pool[1, start:start + L])
    j = np.arange(L)
    bt = np.asarray(block_table[b].cpu().numpy() if hasattr(block_table, "cpu") else block_table[b])
    pool = kv_pool.detach().cpu()
    return pool[bt[j // page_size], 1, j % page_size].float().numpy().astype(np.float32)


def quantize_v(v32: np.ndarray):
    """V fp32 [L, Hkv, D] -> (codes uint8 [ntiles, Hkv, D, 128], scales fp32 [Hkv, D]):
    per channel scale = amax / 448, code = e4m3(v * (448 / amax)), keys innermost,
    zero codes past L."""
    L, H, D = v32.shape
    amax = _amax(v32, axis=0)
    nt = (L + V_TILE - 1) // V_TILE
    c = np.zeros((nt * V_TILE, H, D), dtype=np.uint8)
    c[:L] = _codes(v32, _inv_scale(amax)[None])
    return np.ascontiguousarray(c.reshape(nt, V_TILE, H, D).transpose(0, 2, 3, 1)), _scale(amax)


def dequantize_v(codes: np.ndarray, scale: np.ndarray, L: int) -> np.ndarray:
    """Inverse layout of :func:`quantize_v`: float64 [L, Hkv, D]."""
    nt, H, D, _ = codes.shape
    vals = e4m3_values(codes.transpose(0, 3, 1, 2).reshape(nt * V_TILE, H, D))[:L]
    return vals * scale.astype(np.float64)[None]


def attention_fp8(wl, rows=None):
    """The fp8 P.V method against the float64 attention over the dequantised
    Q, K and V: returns (out, bound), both [n, Hq, D].

    ``out`` is softmax(scale * q^ . k^) v^ with the exact softmax. The method
    also rounds each probability to e4m3: with p relative to the row max,
    the coded value p * 2^(2 + d), d >= 0 (a running max that trails the row
    max; no code above 2^8, so none saturates), is within 2^-4 of it relatively
    or 2^-10 absolutely, i.e. 2^-12 in units of p, so the output moves by at
    most (2^-4 sum p |v^| + 2^-12 sum |v^|) / sum p; ``bound`` is that plus
    the bf16 rounding of the output (2^-8 |out|) and 1e-4 for fp32 sums and
    exp2 approximations.
    """
    cu = wl.cu_q.numpy().astype(np.int64)
    sl = wl.seq_lens.numpy().astype(np.int64)
    starts = np.concatenate([[0], np.cumsum(sl)])
    toks = np.arange(int(cu[-1])) if rows is None else np.asarray(list(rows), dtype=np.int64)
    G = wl.n_heads_q // wl.n_heads_kv
    qc, qs = quantize_q(_bf16_to_f32(wl.q[torch_index(toks)]))
    q_deq = e4m3_values(qc) * qs.astype(np.float64)[:, :, None]
    seq_of = np.searchsorted(cu, toks, side="right") - 1
    out = np.zeros((len(toks), wl.n_heads_q, wl.head_dim), dtype=np.float64)
    bound = np.zeros_like(out)
    for b in np.unique(seq_of):
        b = int(b)
        L = int(sl[b])
        ql = int(cu[b + 1] - cu[b])
        k32 = logical_k(wl.kv_pool, wl.block_table, wl.seq_lens, b, wl.page_size, int(starts[b]))
        kc, ks = quantize_k(k32, k_mean(k32))
        vc, vs = quantize_v(logical_v(wl.kv_pool, wl.block_table, wl.seq_lens, b, wl.page_size,
                                      int(starts[b])))
        v_deq = dequantize_v(vc, vs, L)
        mine = np.nonzero(seq_of == b)[0]
        for hk in range(wl.n_heads_kv):
            k = e4m3_values(kc[:L, hk]) * np.repeat(ks[:, hk].astype(np.float64), 64)[:L, None]
            vh = v_deq[:, hk]
            for n in mine:
                pos = L - ql + (int(toks[n]) - int(cu[b]))
                nk = min(L, pos + 1) if wl.causal else L
                if nk <= 0:
                    continue
                for h in range(hk * G, (hk + 1) * G):
                    s = (k[:nk] @ q_deq[n, h]) * wl.scale
                    w = np.exp(s - s.max())
                    o = (w @ vh[:nk]) / w.sum()
                    out[n, h] = o
                    bound[n, h] = ((2.0 ** -4) * (w @ np.abs(vh[:nk]))
                                   + (2.0 ** -(10 + P_SCALE_LOG2)) * np.abs(vh[:nk]).sum(0)) \
                        / w.sum() + (2.0 ** -8) * np.abs(o) + 1e-4
    return out, bound
