"""Pins for the oracle's cache write (CPU only): the ``kv_write`` node of the
GB10 model graph (``reshape_and_cache_flash``) in front of attention.

A hand-placed slot, a dense attention over logical K/V rebuilt independently
(the new rows overwrite the last ql_b logical keys), the pos < 0 rule and the
contiguous layout.
"""
import math

import numpy as np
import torch

import oracle
import workloads


def _pool(pages, hkv, d, P=64, fill=0.0):
    return torch.full((pages, 2, P, hkv, d), fill, dtype=torch.bfloat16)


def test_slot_of_each_new_token():
    # one sequence, L = 70, three new tokens: positions 67, 68, 69 = logical
    # slot 1 (page 5 here), rows 3, 4, 5
    pool = _pool(8, 1, 8)
    bt = torch.tensor([[2, 5]], dtype=torch.int32)
    sl = torch.tensor([70], dtype=torch.int32)
    cu = torch.tensor([0, 3], dtype=torch.int32)
    k = torch.arange(3 * 8, dtype=torch.float32).reshape(3, 1, 8).to(torch.bfloat16) + 1
    v = -k
    out = oracle.append_kv(pool, bt, sl, cu, k, v)
    expect = pool.clone()
    for i in range(3):
        expect[5, 0, 3 + i] = k[i]
        expect[5, 1, 3 + i] = v[i]
    assert torch.equal(out.view(torch.int16), expect.view(torch.int16))
    assert torch.equal(pool, _pool(8, 1, 8))  # the input is not modified


def test_tokens_without_a_slot_are_skipped():
    # ql = 5 > L = 3: tokens 0 and 1 have positions -2, -1
    pool = _pool(4, 2, 8, fill=7.0)
    bt = torch.tensor([[1]], dtype=torch.int32)
    sl = torch.tensor([3], dtype=torch.int32)
    cu = torch.tensor([0, 5], dtype=torch.int32)
    k = torch.randn(5, 2, 8).to(torch.bfloat16)
    v = torch.randn(5, 2, 8).to(torch.bfloat16)
    out = oracle.append_kv(pool, bt, sl, cu, k, v)
    expect = pool.clone()
    for i in range(2, 5):
        expect[1, 0, i - 2] = k[i]
        expect[1, 1, i - 2] = v[i]
    assert torch.equal(out.view(torch.int16), expect.view(torch.int16))


def test_contiguous_rows():
    wl = workloads.make_contiguous("c", 11, [2, 3], [5, 9], 4, 2, 128, causal=True)
    k, v = workloads.new_kv_rows(wl, 3)
    out = oracle.append_kv(wl.kv_pool, None, wl.seq_lens, wl.cu_q, k, v)
    expect = wl.kv_pool.clone()
    # sequence 0: rows 3, 4 (tokens 0, 1); sequence 1 starts at row 5: rows 5+6..5+8
    for t, row in ((0, 3), (1, 4), (2, 11), (3, 12), (4, 13)):
        expect[0, row] = k[t]
        expect[1, row] = v[t]
    assert torch.equal(out.view(torch.int16), expect.view(torch.int16))


def _dense(q, K, V, ql, L, scale, causal, hq, hkv):
    """Dense attention of one sequence in float64 (einsum, explicit mask)."""
    G = hq // hkv
    qh = q.reshape(ql, hkv, G, -1)
    s = np.einsum("tkgd,jkd->tkgj", qh, K) * scale
    pos = L - ql + np.arange(ql)
    mask = np.arange(L)[None, :] <= pos[:, None] if causal else np.ones((ql, L), bool)
    s = np.where(mask[:, None, None, :], s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(s - m)
    den = w.sum(-1, keepdims=True)
    o = np.einsum("tkgj,jkd->tkgd", w, V) / np.where(den > 0, den, 1.0)
    return o.reshape(ql, hq, -1)


def test_attention_over_the_appended_cache_matches_dense():
    wl = workloads.make_paged("a", 21, [1, 4, 3], [40, 130, 64], 8, 2, 128, causal=True, extra_pages=2)
    k, v = workloads.new_kv_rows(wl, 5)
    wl2 = oracle.append_workload(wl, k, v)
    got, _ = oracle.forward_workload(wl2)
    pool = wl.kv_pool.float().numpy().astype(np.float64)  # the ORIGINAL pool
    bt = wl.block_table.numpy()
    cu = wl.cu_q.numpy()
    q = wl.q.float().numpy().astype(np.float64)
    kn = k.float().numpy().astype(np.float64)
    vn = v.float().numpy().astype(np.float64)
    for b in range(wl.num_seqs):
        L = int(wl.seq_lens[b])
        ql = int(cu[b + 1] - cu[b])
        j = np.arange(L)
        K = pool[bt[b, j // 64], 0, j % 64].copy()
        V = pool[bt[b, j // 64], 1, j % 64].copy()
        K[L - ql:] = kn[cu[b]:cu[b + 1]]  # the new tokens are the last ql keys
        V[L - ql:] = vn[cu[b]:cu[b + 1]]
        ref = _dense(q[cu[b]:cu[b + 1]], K, V, ql, L, wl.scale, True, wl.n_heads_q, wl.n_heads_kv)
        assert np.abs(got[cu[b]:cu[b + 1]] - ref).max() < 1e-12
    # and the write matters: the old cache gives a different answer
    old, _ = oracle.forward_workload(wl)
    assert np.abs(old - got).max() > 1e-3
