"""Float64 CPU oracle for paged-KV varlen attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares nothing with the CUDA library:
the arithmetic lives in ``pattn_oracle.c`` (plain C, double precision,
pthreads), built here with gcc.

Functions:

* :func:`forward` -- attention output and log-sum-exp for every query token
  (or a chosen subset of tokens), for a key window if asked.
* :func:`combine` -- log-sum-exp merge of results over disjoint key sets.
* :func:`append_kv` -- the cache write in front of attention (the GB10 model
  graph's ``kv_write`` node, ``reshape_and_cache_flash``): the new tokens' K and
  V rows into their cache slots, as a fresh pool. Plain numpy indexing.

Both are pinned by the ``-m "not gpu"`` tests against closed forms, a dense
brute force written separately in numpy, and invariants (page permutation,
K offset, GQA = MHA with repeated heads, split identity).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pattn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to the source (gcc, -O2, no FP contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.pattn_oracle_forward.restype = ctypes.c_int
            lib.pattn_oracle_forward.argtypes = [
                vp, vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i32, i32,
                i64, i64, i64, i64, dbl, i32, vp, i64, i64, i64, i32]
            lib.pattn_oracle_combine.restype = None
            lib.pattn_oracle_combine.argtypes = [vp, vp, vp, vp, i32, i64, i32]
            lib.pattn_oracle_threads.restype = ctypes.c_int
            lib.pattn_oracle_threads.argtypes = []
            _lib = lib
    return _lib


def threads() -> int:
    """Host threads the oracle uses by default (online processors)."""
    return int(_load().pattn_oracle_threads())


def _bits(t) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 numpy array of the bits."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(t) -> np.ndarray:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return np.ascontiguousarray(t, dtype=np.int32)
    return np.ascontiguousarray(t.detach().cpu().numpy().astype(np.int32))


def pool_strides(n_heads_kv: int, head_dim: int, page_size: int, layout: str = "paged",
                 rows: int = 0) -> Tuple[int, int, int, int]:
    """Element strides (page, K/V, row, head) of the supported cache layouts.

    * ``paged``: ``[page][2][P][Hkv][D]`` (K and V as separate 64-row blocks of a page)
    * ``paged_interleaved``: ``[page][2][P][Hkv][2][D]`` -- K and V interleaved per
      head, as in the trtllm-gen decode manifest's 6-D ``kv`` buffer; the outer 2
      is a second slice the oracle does not read.
    * ``contiguous``: ``[2][rows][Hkv][D]``.
    """
    D, H, P = head_dim, n_heads_kv, page_size
    if layout == "paged":
        return (2 * P * H * D, P * H * D, H * D, D)
    if layout == "paged_interleaved":
        return (2 * P * H * 2 * D, D, H * 2 * D, 2 * D)
    if layout == "contiguous":
        return (0, rows * H * D, H * D, D)
    raise ValueError(layout)


def forward(q, kv_pool, block_table, seq_lens, cu_q, n_heads_q: int, n_heads_kv: int,
            head_dim: int, page_size: int, scale: float, causal: bool,
            rows: Optional[Sequence[int]] = None, key_window: Optional[Tuple[int, int]] = None,
            strides: Optional[Tuple[int, int, int, int]] = None, n_threads: int = 0,
            want_lse: bool = True):
    """Attention in float64. Returns ``(out [n_rows, Hq, D], lse [n_rows, Hq])``.

    ``rows`` selects query tokens (global indices into ``q``); ``None`` = all.
    ``key_window = (j0, j1)`` keeps only logical keys ``j0 <= j < j1`` of every
    sequence (``j1 < 0``: no upper bound), used to check the split-KV merge.
    """
    lib = _load()
    qb = _bits(q)
    kvb = _bits(kv_pool)
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    cq = _i32(cu_q)
    total_q = qb.shape[0]
    if strides is None:
        if bt is not None:
            strides = pool_strides(n_heads_kv, head_dim, page_size, "paged")
        else:
            strides = pool_strides(n_heads_kv, head_dim, page_size, "contiguous", kvb.shape[1])
    if rows is None:
        rows_arr = None
        n_rows = total_q
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = rows_arr.shape[0]
    out = np.zeros((n_rows, n_heads_q, head_dim), dtype=np.float64)
    lse = np.zeros((n_rows, n_heads_q), dtype=np.float64) if want_lse else None
    if n_rows == 0:
        return out, lse
    j0, j1 = key_window if key_window is not None else (0, -1)
    p = lambda a: a.ctypes.data if a is not None else None
    rc = lib.pattn_oracle_forward(
        p(out), p(lse), p(qb), p(kvb), p(bt), int(bt.shape[1]) if bt is not None else 0,
        p(sl), p(cq), int(sl.shape[0]), n_heads_q, n_heads_kv, head_dim, page_size,
        int(strides[0]), int(strides[1]), int(strides[2]), int(strides[3]),
        float(scale), int(bool(causal)), p(rows_arr), int(n_rows), int(j0), int(j1), int(n_threads))
    if rc != 0:
        raise RuntimeError(f"pattn_oracle_forward failed with {rc}")
    return out, lse


def forward_workload(wl, rows=None, key_window=None, n_threads: int = 0):
    """:func:`forward` on a :class:`workloads.Workload`."""
    return forward(wl.q, wl.kv_pool, wl.block_table, wl.seq_lens, wl.cu_q, wl.n_heads_q,
                   wl.n_heads_kv, wl.head_dim, wl.page_size, wl.scale, wl.causal,
                   rows=rows, key_window=key_window, n_threads=n_threads)


def combine(out_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge ``out_parts [S, n, D]`` / ``lse_parts [S, n]`` -> ``(out [n, D], lse [n])``."""
    lib = _load()
    op = np.ascontiguousarray(out_parts, dtype=np.float64)
    lp = np.ascontiguousarray(lse_parts, dtype=np.float64)
    S, n, d = op.shape
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    lib.pattn_oracle_combine(out.ctypes.data, lse.ctypes.data, op.ctypes.data, lp.ctypes.data,
                             int(S), int(n), int(d))
    return out, lse


def append_kv(kv_pool, block_table, seq_lens, cu_q, k_new, v_new, page_size: int = 64):
    """The cache write of the GB10 model graph's ``kv_write`` node
    (``reshape_and_cache_flash``, "k:write,v:write", "cache bf16"), on a copy.

    Token i of sequence b (``i < ql_b = cu_q[b+1] - cu_q[b]``) is the key at
    logical position ``pos = seq_lens[b] - ql_b + i`` (the new tokens are the
    last ``ql_b`` keys, the same bottom-right alignment as the attention); its
    K and V rows ``k_new[t]``, ``v_new[t]`` (``t = cu_q[b] + i``, shape
    ``[Hkv, D]``) go to row ``pos % P`` of page ``block_table[b][pos // P]``,
    or, with ``block_table = None``, to row ``sum(seq_lens[:b]) + pos`` of the
    K and V planes. Tokens with ``pos < 0`` have no slot and are skipped.
    Returns the new pool (bf16 tensor on the CPU); the input is not modified.
    """
    import torch
    pool = kv_pool.detach().cpu().clone()
    kn = k_new.detach().cpu()
    vn = v_new.detach().cpu()
    sl = _i32(seq_lens)
    cq = _i32(cu_q)
    bt = _i32(block_table)
    start = 0
    for b in range(sl.shape[0]):
        L = int(sl[b])
        q0, q1 = int(cq[b]), int(cq[b + 1])
        ql = q1 - q0
        for i in range(ql):
            pos = L - ql + i
            if pos < 0:
                continue
            t = q0 + i
            if bt is None:
                pool[0, start + pos] = kn[t]
                pool[1, start + pos] = vn[t]
            else:
                page = int(bt[b, pos // page_size])
                pool[page, 0, pos % page_size] = kn[t]
                pool[page, 1, pos % page_size] = vn[t]
        start += L
    return pool


def append_workload(wl, k_new, v_new):
    """:func:`append_kv` on a :class:`workloads.Workload`: the same workload with
    the updated pool."""
    import dataclasses
    pool = append_kv(wl.kv_pool, wl.block_table, wl.seq_lens, wl.cu_q, k_new, v_new, wl.page_size)
    return dataclasses.replace(wl, kv_pool=pool)
