"""paged_kv_flashattention_varlen_gb300 -- paged-KV varlen attention for GB300.

Python face of ``libpattn.so``. The functions below check tensor types and
pass raw pointers and the current CUDA stream to the C ABI (include/pattn.h);
PyTorch only provides device memory and streams. There is no CPU path.

    forward(out, q, kv_pool, block_table, seq_lens, cu_q, *, max_q, max_kv,
            n_heads_kv, scale, causal, num_pages=None, stream=None)
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

from . import _lib

__all__ = ["PattnError", "forward", "forward_append", "forward_fp8qk", "quantize_qk", "forward_fp8",
           "quantize_v", "forward_noalloc",
           "forward_host", "workspace_size",
           "set_workspace", "device_status", "status_string", "selftest_wait_timeout",
           "selftest_attention_timeout", "plan_items",
           "profile_enable",
           "profile_read",
           "profile_read_kernels", "STATUS", "library_path"]

STATUS = {
    0: "PATTN_OK", 1: "PATTN_ERR_INVALID_ARG", 2: "PATTN_ERR_UNSUPPORTED", 3: "PATTN_ERR_CUDA",
    4: "PATTN_ERR_NO_MEMORY", 5: "PATTN_ERR_DEVICE_BAD_INPUT", 6: "PATTN_ERR_DEVICE_TIMEOUT",
}


class PattnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS.get(code, code)} ({status_string(code)})")


def library_path() -> str:
    return _lib.LIB_PATH


def status_string(code: int) -> str:
    return _lib.load().pattn_status_string(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != 0:
        raise PattnError(code, where)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _shape_args(q, kv_pool, block_table, n_heads_kv: int, num_pages: Optional[int]):
    total_q, n_heads_q, head_dim = (int(x) for x in q.shape)
    if block_table is not None:
        page_size = int(kv_pool.shape[2])
        pages = int(kv_pool.shape[0]) if num_pages is None else int(num_pages)
    else:
        page_size = 64
        pages = int(kv_pool.shape[1]) if num_pages is None else int(num_pages)
    return total_q, n_heads_q, head_dim, page_size, pages


def forward(out, q, kv_pool, block_table, seq_lens, cu_q, *, max_q: int, max_kv: int,
            n_heads_kv: int, scale: float, causal: bool, num_pages: Optional[int] = None,
            stream=None, check: bool = True) -> int:
    """Attention over a paged KV cache on the GPU (``pattn_forward``).

    ``q``/``out``: bf16 [total_q, Hq, D] on the device; ``kv_pool``: bf16
    [pages, 2, 64, Hkv, D] (or [2, rows, Hkv, D] with ``block_table=None``);
    ``block_table`` int32 [B, ceil(max_kv/64)]; ``seq_lens`` int32 [B];
    ``cu_q`` int32 [B+1]. Returns the status code (raises if ``check``).
    """
    import torch
    for name, t, dt in (("out", out, torch.bfloat16), ("q", q, torch.bfloat16),
                        ("kv_pool", kv_pool, torch.bfloat16), ("seq_lens", seq_lens, torch.int32),
                        ("cu_q", cu_q, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name}: expected a contiguous CUDA {dt} tensor")
    if block_table is not None and (block_table.dtype != torch.int32 or not block_table.is_cuda
                                    or not block_table.is_contiguous()):
        raise TypeError("block_table: expected a contiguous CUDA int32 tensor or None")
    total_q, hq, d, page, pages = _shape_args(q, kv_pool, block_table, n_heads_kv, num_pages)
    rc = _lib.load().pattn_forward(
        _ptr(out), _ptr(q), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens), _ptr(cu_q),
        int(seq_lens.numel()), total_q, int(max_q), int(max_kv), hq, int(n_heads_kv), d, page,
        pages, float(scale), int(bool(causal)), _stream_handle(stream))
    if check:
        _check(rc, "pattn_forward")
    return rc


def forward_append(out, q, k_new, v_new, kv_pool, block_table, seq_lens, cu_q, *, max_q: int,
                   max_kv: int, n_heads_kv: int, scale: float, causal: bool,
                   num_pages: Optional[int] = None, stream=None, check: bool = True) -> int:
    """Cache write of the new tokens, then attention (``pattn_forward_append``).

    ``k_new``/``v_new``: bf16 [total_q, Hkv, D] on the device, the K and V rows of
    the query tokens; token i of sequence b is written to cache position
    ``seq_lens[b] - ql_b + i`` of ``kv_pool`` (in place), then the attention reads
    the updated cache. Other arguments as for :func:`forward`.
    """
    import torch
    for name, t, dt in (("out", out, torch.bfloat16), ("q", q, torch.bfloat16),
                        ("k_new", k_new, torch.bfloat16), ("v_new", v_new, torch.bfloat16),
                        ("kv_pool", kv_pool, torch.bfloat16), ("seq_lens", seq_lens, torch.int32),
                        ("cu_q", cu_q, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name}: expected a contiguous CUDA {dt} tensor")
    if block_table is not None and (block_table.dtype != torch.int32 or not block_table.is_cuda
                                    or not block_table.is_contiguous()):
        raise TypeError("block_table: expected a contiguous CUDA int32 tensor or None")
    total_q, hq, d, page, pages = _shape_args(q, kv_pool, block_table, n_heads_kv, num_pages)
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if tuple(t.shape) != (total_q, int(n_heads_kv), d):
            raise ValueError(f"{name}: expected shape {(total_q, int(n_heads_kv), d)}, got {tuple(t.shape)}")
    rc = _lib.load().pattn_forward_append(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens),
        _ptr(cu_q), int(seq_lens.numel()), total_q, int(max_q), int(max_kv), hq, int(n_heads_kv), d,
        page, pages, float(scale), int(bool(causal)), _stream_handle(stream))
    if check:
        _check(rc, "pattn_forward_append")
    return rc


def _check_device_args(out, q, kv_pool, block_table, seq_lens, cu_q):
    import torch
    for name, t, dt in (("out", out, torch.bfloat16), ("q", q, torch.bfloat16),
                        ("kv_pool", kv_pool, torch.bfloat16), ("seq_lens", seq_lens, torch.int32),
                        ("cu_q", cu_q, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name}: expected a contiguous CUDA {dt} tensor")
    if block_table is not None and (block_table.dtype != torch.int32 or not block_table.is_cuda
                                    or not block_table.is_contiguous()):
        raise TypeError("block_table: expected a contiguous CUDA int32 tensor or None")


def forward_fp8qk(out, q, kv_pool, block_table, seq_lens, cu_q, *, max_q: int, max_kv: int,
                  n_heads_kv: int, scale: float, causal: bool, num_pages: Optional[int] = None,
                  stream=None, check: bool = True) -> int:
    """Quantised-QK attention (``pattn_forward_fp8qk``): K smoothed by its mean,
    Q and K as e4m3 codes with row / 64-key block scales, PV in bf16. head_dim 128.
    Arguments as for :func:`forward`."""
    _check_device_args(out, q, kv_pool, block_table, seq_lens, cu_q)
    total_q, hq, d, page, pages = _shape_args(q, kv_pool, block_table, n_heads_kv, num_pages)
    rc = _lib.load().pattn_forward_fp8qk(
        _ptr(out), _ptr(q), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens), _ptr(cu_q),
        int(seq_lens.numel()), total_q, int(max_q), int(max_kv), hq, int(n_heads_kv), d, page,
        pages, float(scale), int(bool(causal)), _stream_handle(stream))
    if check:
        _check(rc, "pattn_forward_fp8qk")
    return rc


def quantize_qk(q, kv_pool, block_table, seq_lens, cu_q, *, max_q: int, max_kv: int,
                n_heads_kv: int, num_pages: Optional[int] = None, stream=None):
    """The e4m3 codes and scales of :func:`forward_fp8qk` (``pattn_quantize_qk``).

    Returns ``(q8 uint8 [T, Hq, D], q_scale f32 [T, Hq], k8 uint8 [B * nb, 64, Hkv, D],
    k_scale f32 [B * nb, Hkv])`` with ``nb = 2 * ceil(max_kv / 128)``; block j of
    sequence b is ``b * nb + j``."""
    import torch
    total_q, hq, d, page, pages = _shape_args(q, kv_pool, block_table, n_heads_kv, num_pages)
    B = int(seq_lens.numel())
    nb = 2 * max(1, -(-int(max_kv) // 128))
    dev = q.device
    q8 = torch.zeros((total_q, hq, d), dtype=torch.uint8, device=dev)
    qs = torch.zeros((total_q, hq), dtype=torch.float32, device=dev)
    k8 = torch.zeros((B * nb, 64, int(n_heads_kv), d), dtype=torch.uint8, device=dev)
    ks = torch.zeros((B * nb, int(n_heads_kv)), dtype=torch.float32, device=dev)
    rc = _lib.load().pattn_quantize_qk(
        _ptr(q8), _ptr(qs), _ptr(k8), _ptr(ks), _ptr(q), _ptr(kv_pool), _ptr(block_table),
        _ptr(seq_lens), _ptr(cu_q), B, total_q, int(max_q), int(max_kv), hq, int(n_heads_kv), d, page,
        pages, _stream_handle(stream))
    _check(rc, "pattn_quantize_qk")
    return q8, qs, k8, ks


def forward_fp8(out, q, kv_pool, block_table, seq_lens, cu_q, *, max_q: int, max_kv: int,
                n_heads_kv: int, scale: float, causal: bool, num_pages: Optional[int] = None,
                stream=None, check: bool = True) -> int:
    """fp8 attention (``pattn_forward_fp8``): Q, K (mean-smoothed), P and V as
    e4m3 codes, S and P.V on e4m3 tensor cores. head_dim 128. Arguments as for
    :func:`forward`."""
    _check_device_args(out, q, kv_pool, block_table, seq_lens, cu_q)
    total_q, hq, d, page, pages = _shape_args(q, kv_pool, block_table, n_heads_kv, num_pages)
    rc = _lib.load().pattn_forward_fp8(
        _ptr(out), _ptr(q), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens), _ptr(cu_q),
        int(seq_lens.numel()), total_q, int(max_q), int(max_kv), hq, int(n_heads_kv), d, page,
        pages, float(scale), int(bool(causal)), _stream_handle(stream))
    if check:
        _check(rc, "pattn_forward_fp8")
    return rc


def quantize_v(q, kv_pool, block_table, seq_lens, cu_q, *, max_q: int, max_kv: int,
               n_heads_kv: int, num_pages: Optional[int] = None, stream=None):
    """The e4m3 V codes and per-channel scales of :func:`forward_fp8`
    (``pattn_quantize_v``; ``q`` gives the shapes only).

    Returns ``(v8 uint8 [B * nt, Hkv, D, 128], v_scale f32 [B, Hkv, D])`` with
    ``nt = ceil(max_kv / 128)``; 128-key tile t of sequence b is ``b * nt + t``,
    keys innermost."""
    import torch
    total_q, hq, d, page, pages = _shape_args(q, kv_pool, block_table, n_heads_kv, num_pages)
    B = int(seq_lens.numel())
    nt = max(1, -(-int(max_kv) // 128))
    dev = q.device
    v8 = torch.zeros((B * nt, int(n_heads_kv), d, 128), dtype=torch.uint8, device=dev)
    vs = torch.zeros((B, int(n_heads_kv), d), dtype=torch.float32, device=dev)
    rc = _lib.load().pattn_quantize_v(
        _ptr(v8), _ptr(vs), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens), _ptr(cu_q), B, total_q,
        int(max_q), int(max_kv), hq, int(n_heads_kv), d, page, pages, _stream_handle(stream))
    _check(rc, "pattn_quantize_v")
    return v8, vs


def forward_noalloc(out, q, kv_pool, block_table, seq_lens, cu_q, *, max_q: int, max_kv: int,
                    n_heads_kv: int, scale: float, causal: bool, num_pages: Optional[int] = None,
                    stream=None, check: bool = True) -> int:
    """As :func:`forward`, through ``pattn_forward_noalloc``: no device allocation, the
    library's fixed scratch instead of its workspace (for callers that must not
    allocate; calls sharing the scratch must not overlap on the GPU)."""
    import torch
    for name, t, dt in (("out", out, torch.bfloat16), ("q", q, torch.bfloat16),
                        ("kv_pool", kv_pool, torch.bfloat16), ("seq_lens", seq_lens, torch.int32),
                        ("cu_q", cu_q, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name}: expected a contiguous CUDA {dt} tensor")
    total_q, hq, d, page, pages = _shape_args(q, kv_pool, block_table, n_heads_kv, num_pages)
    rc = _lib.load().pattn_forward_noalloc(
        _ptr(out), _ptr(q), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens), _ptr(cu_q),
        int(seq_lens.numel()), total_q, int(max_q), int(max_kv), hq, int(n_heads_kv), d, page,
        pages, float(scale), int(bool(causal)), _stream_handle(stream))
    if check:
        _check(rc, "pattn_forward_noalloc")
    return rc


def forward_host(out, q, kv_pool, block_table, seq_lens, cu_q, *, max_q: int, max_kv: int,
                 n_heads_kv: int, scale: float, causal: bool, num_pages: Optional[int] = None,
                 stream=None) -> None:
    """End-to-end call on HOST tensors (``pattn_forward_host``): copies in, runs, copies out."""
    import torch
    for name, t in (("out", out), ("q", q), ("kv_pool", kv_pool), ("seq_lens", seq_lens),
                    ("cu_q", cu_q)):
        if t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name}: expected a contiguous host tensor")
    total_q, hq, d, page, pages = _shape_args(q, kv_pool, block_table, n_heads_kv, num_pages)
    rc = _lib.load().pattn_forward_host(
        _ptr(out), _ptr(q), _ptr(kv_pool), kv_pool.numel() * kv_pool.element_size(),
        _ptr(block_table), _ptr(seq_lens), _ptr(cu_q), int(seq_lens.numel()), total_q, int(max_q),
        int(max_kv), hq, int(n_heads_kv), d, page, pages, float(scale), int(bool(causal)),
        _stream_handle(stream))
    _check(rc, "pattn_forward_host")


def workspace_size(num_seqs: int, total_q: int, max_q: int, max_kv: int, n_heads_q: int,
                   n_heads_kv: int, head_dim: int, page_size: int = 64) -> int:
    return int(_lib.load().pattn_workspace_size(num_seqs, total_q, max_q, max_kv, n_heads_q,
                                                n_heads_kv, head_dim, page_size))


def set_workspace(buf=None) -> None:
    """Use a caller-owned CUDA byte tensor as the workspace (None: library-owned)."""
    if buf is None:
        _check(_lib.load().pattn_set_workspace(None, 0), "pattn_set_workspace")
    else:
        _check(_lib.load().pattn_set_workspace(_ptr(buf), buf.numel() * buf.element_size()),
               "pattn_set_workspace")


def device_status(stream=None) -> int:
    """Synchronise, read and clear the device error word (0 = fine)."""
    return int(_lib.load().pattn_get_device_status(_stream_handle(stream)))


def selftest_wait_timeout(stream=None) -> None:
    """Launch the failure-detection self-test (``pattn_selftest_wait_timeout``):
    a bounded wait that runs out after its limit and sets the timeout bit that
    :func:`device_status` then reports."""
    _check(_lib.load().pattn_selftest_wait_timeout(_stream_handle(stream)), "pattn_selftest_wait_timeout")


def selftest_attention_timeout(out, q, kv_pool, block_table, seq_lens, cu_q, *, max_q: int, max_kv: int,
                               n_heads_kv: int, scale: float, causal: bool,
                               num_pages: Optional[int] = None, stream=None) -> None:
    """Launch the attention kernels' failure-detection self-test
    (``pattn_selftest_attention_timeout``): :func:`forward` on this batch with
    the first CTA's MMA-issuing thread made to wait on a phase that nothing
    completes, so that its bounded wait runs out and the CTA takes its
    abort-and-drain path; :func:`device_status` then reports the timeout."""
    import torch
    for name, t, dt in (("out", out, torch.bfloat16), ("q", q, torch.bfloat16),
                        ("kv_pool", kv_pool, torch.bfloat16), ("seq_lens", seq_lens, torch.int32),
                        ("cu_q", cu_q, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name}: expected a contiguous CUDA {dt} tensor")
    total_q, hq, d, page, pages = _shape_args(q, kv_pool, block_table, n_heads_kv, num_pages)
    _check(_lib.load().pattn_selftest_attention_timeout(
        _ptr(out), _ptr(q), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens), _ptr(cu_q),
        int(seq_lens.numel()), total_q, int(max_q), int(max_kv), hq, int(n_heads_kv), d, page,
        pages, float(scale), int(bool(causal)), _stream_handle(stream)), "pattn_selftest_attention_timeout")


def plan_items(block_table, seq_lens, cu_q, *, total_q: int, max_q: int, max_kv: int, n_heads_q: int,
               n_heads_kv: int, head_dim: int, causal: bool, num_pages: int, capacity: int = 1 << 16,
               stream=None):
    """The tile plan of a batch (``pattn_plan_items``): runs only the device-side
    planner and returns (prefill items, decode items, counts) as numpy int32
    arrays, items [n, 4] = (sequence | split << 24, kv_head << 16 | q tile,
    first KV tile << 16 | end KV tile, first partial row or -1) in list order,
    counts = (prefill items, decode items, split units, partial rows)."""
    import numpy as np
    import torch
    for name, t in (("seq_lens", seq_lens), ("cu_q", cu_q)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name}: expected a contiguous CUDA int32 tensor")
    pre = np.zeros((capacity, 4), dtype=np.int32)
    dec = np.zeros((capacity, 4), dtype=np.int32)
    counts = np.zeros(4, dtype=np.int32)
    rc = _lib.load().pattn_plan_items(
        _ptr(block_table), _ptr(seq_lens), _ptr(cu_q), int(seq_lens.numel()), int(total_q), int(max_q),
        int(max_kv), int(n_heads_q), int(n_heads_kv), int(head_dim), 64, int(num_pages), int(bool(causal)),
        pre.ctypes.data, dec.ctypes.data, int(capacity), counts.ctypes.data, _stream_handle(stream))
    _check(rc, "pattn_plan_items")
    return pre[:min(int(counts[0]), capacity)], dec[:min(int(counts[1]), capacity)], counts


def profile_enable(on: bool = True) -> None:
    _check(_lib.load().pattn_profile_enable(int(bool(on))), "pattn_profile_enable")


def profile_read_kernels() -> Tuple[Tuple[float, float, float, float, float], int]:
    """((ms plan with the cache write, ms quantisation, ms decode kernel, ms prefill kernel, ms after), calls)."""
    ms = (ctypes.c_double * 5)()
    n = ctypes.c_int()
    _check(_lib.load().pattn_profile_read_kernels(ms, ctypes.byref(n)), "pattn_profile_read_kernels")
    return tuple(ms[i] for i in range(5)), n.value


def profile_read() -> Tuple[float, float, float, int]:
    """(ms plan, ms attention, ms combine, calls) summed since the last read."""
    a, b, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    n = ctypes.c_int()
    _check(_lib.load().pattn_profile_read(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c),
                                          ctypes.byref(n)), "pattn_profile_read")
    return a.value, b.value, c.value, n.value
