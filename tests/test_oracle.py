"""Pins for the float64 oracle (CPU only).

The pages print no attention outputs, so the oracle is pinned to what the
mathematics fixes: closed forms, a dense brute force written separately here
in numpy (einsum + explicit mask + log-sum-exp, not the oracle's token walk),
and invariants a wrong index, sign or dropped term would break.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


# ----------------------------------------------------------------------------
# independent dense reference (numpy): gather the logical cache, then softmax
# ----------------------------------------------------------------------------
def _f64(t):
    return t.float().numpy().astype(np.float64)


def logical_kv(wl, b):
    """Logical K, V [L, Hkv, D] of sequence b, gathered with numpy fancy indexing."""
    L = int(wl.seq_lens[b])
    pool = _f64(wl.kv_pool)
    if wl.block_table is None:
        start = int(wl.seq_lens[:b].sum())
        return pool[0, start:start + L], pool[1, start:start + L]
    j = np.arange(L)
    pages = wl.block_table.numpy()[b, j // wl.page_size]
    rows = j % wl.page_size
    return pool[pages, 0, rows], pool[pages, 1, rows]


def dense_attention(wl):
    q = _f64(wl.q)
    cu = wl.cu_q.numpy().astype(np.int64)
    G = wl.n_heads_q // wl.n_heads_kv
    out = np.zeros_like(q)
    lse = np.full(q.shape[:2], -np.inf)
    for b in range(wl.num_seqs):
        ql = cu[b + 1] - cu[b]
        L = int(wl.seq_lens[b])
        if ql == 0:
            continue
        K, V = logical_kv(wl, b)
        K = np.repeat(K, G, axis=1)
        V = np.repeat(V, G, axis=1)
        Q = q[cu[b]:cu[b + 1]]
        S = np.einsum("ihd,jhd->hij", Q, K) * wl.scale       # [Hq, ql, L]
        i = np.arange(ql)[:, None]
        j = np.arange(L)[None, :]
        vis = np.ones((ql, L), bool) if not wl.causal else (j <= (L - ql + i))
        S = np.where(vis[None], S, -np.inf)
        m = S.max(axis=2, initial=-np.inf, keepdims=True)
        has = np.isfinite(m)
        msafe = np.where(has, m, 0.0)
        W = np.exp(S - msafe)
        den = W.sum(axis=2, keepdims=True)
        O = np.einsum("hij,jhd->ihd", W, V) / np.where(den > 0, den, 1.0).transpose(1, 0, 2)
        O = np.where(has.transpose(1, 0, 2), O, 0.0)
        out[cu[b]:cu[b + 1]] = O
        l = (msafe + np.log(np.where(den > 0, den, 1.0)))[:, :, 0].T
        lse[cu[b]:cu[b + 1]] = np.where(has[:, :, 0].T, l, -np.inf)
    return out, lse


def run_oracle(wl, **kw):
    return oracle.forward_workload(wl, **kw)


def small(seed, q_lens, kv_lens, hq, hkv, d, causal=True, P=64, extra=3, **kw):
    return workloads.make_paged("t", seed, q_lens, kv_lens, hq, hkv, d, P, causal=causal,
                                extra_pages=extra, **kw)


# ----------------------------------------------------------------------------
# brute force agreement
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("d", [16, 128, 256])
@pytest.mark.parametrize("g", [1, 2, 6])
@pytest.mark.parametrize("causal", [True, False])
def test_brute_force_small(d, g, causal):
    hkv = 2 if g != 6 else 1
    wl = small(7 + d + g, [3, 1, 5], [70, 1, 130], hkv * g, hkv, d, causal=causal)
    o, l = run_oracle(wl)
    ro, rl = dense_attention(wl)
    assert np.isfinite(o).all()
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)


EDGES = [1, 63, 64, 65, 127, 128, 129]


@pytest.mark.parametrize("L", EDGES)
def test_edge_lengths(L):
    qls = sorted({1, 63, 64, 65, 127, 128, 129, L})
    qls = [x for x in qls if x <= L]
    wl = small(100 + L, qls, [L] * len(qls), 4, 2, 16, causal=True)
    o, l = run_oracle(wl)
    ro, rl = dense_attention(wl)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)
    # non-causal, query length above the KV length
    wl2 = small(200 + L, [L + 1, 1], [L, L], 4, 2, 16, causal=False)
    o2, _ = run_oracle(wl2)
    ro2, _ = dense_attention(wl2)
    np.testing.assert_allclose(o2, ro2, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------
def test_zero_query_gives_mean_of_visible_values():
    wl = small(1, [4], [9], 2, 1, 16, causal=True)
    wl.q.zero_()
    o, l = run_oracle(wl)
    K, V = logical_kv(wl, 0)
    L, ql = 9, 4
    for i in range(ql):
        n = L - ql + i + 1
        np.testing.assert_allclose(o[i, 0], V[:n, 0].mean(axis=0), rtol=0, atol=1e-14)
        np.testing.assert_allclose(l[i, 0], math.log(n), rtol=0, atol=1e-14)


def test_constant_values_give_that_value():
    wl = small(2, [3], [77], 2, 1, 16, causal=False)
    v = torch.randn(16, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    tbl = wl.block_table.numpy()[0]
    for j in range(77):
        wl.kv_pool[tbl[j // 64], 1, j % 64, 0] = v
    o, _ = run_oracle(wl)
    for i in range(3):
        np.testing.assert_allclose(o[i, :], np.broadcast_to(v.float().numpy(), (2, 16)), rtol=0, atol=1e-14)


def test_one_hot_scores_select_one_row():
    # K row j = 8 e_j, q = 8 e_t, scale 1: s_t = 64, every other score 0, so the
    # weight of any other row is e^-64 (about 1.6e-28) of the selected one.
    d, L = 16, 16
    wl = small(4, [1] * L, [L] * L, 1, 1, d, causal=False)
    tbl = wl.block_table.numpy()
    for b in range(L):
        for j in range(L):
            k = torch.zeros(d)
            k[j] = 8.0
            wl.kv_pool[tbl[b, 0], 0, j, 0] = k.to(torch.bfloat16)
        qq = torch.zeros(d)
        qq[b] = 8.0
        wl.q[b, 0] = qq.to(torch.bfloat16)
    wl.scale = 1.0
    o, l = run_oracle(wl)
    for b in range(L):
        K, V = logical_kv(wl, b)
        np.testing.assert_allclose(o[b, 0], V[b, 0], rtol=0, atol=1e-25 * (1 + np.abs(V).max()) * L)
        np.testing.assert_allclose(l[b, 0], 64.0, rtol=0, atol=1e-12)


def test_single_key_returns_its_value_exactly():
    wl = small(5, [1, 1], [1, 1], 6, 2, 128, causal=True)
    o, l = run_oracle(wl)
    for b in range(2):
        K, V = logical_kv(wl, b)
        for h in range(6):
            assert np.array_equal(o[b, h], V[0, h // 3])
            np.testing.assert_allclose(l[b, h], wl.scale * float(_f64(wl.q)[b, h] @ K[0, h // 3]), atol=1e-12)


def test_decode_single_query_causal_equals_noncausal():
    wl = small(6, [1, 1, 1], [5, 64, 200], 8, 2, 128, causal=True)
    o1, l1 = run_oracle(wl)
    wl.causal = False
    o2, l2 = run_oracle(wl)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_no_visible_key_gives_zero():
    # L = 0, and causal rows before the first key (ql > L).
    wl = small(8, [2, 5], [0, 3], 2, 1, 16, causal=True)
    o, l = run_oracle(wl)
    assert np.all(o[:2] == 0) and np.all(np.isneginf(l[:2]))
    assert np.all(o[2:4] == 0) and np.all(np.isneginf(l[2:4]))   # p = 3-5+i < 0 for i < 2
    assert np.all(np.isfinite(l[4:]))
    ro, rl = dense_attention(wl)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# invariants
# ----------------------------------------------------------------------------
def test_page_permutation_invariance_is_bitwise():
    wl = small(9, [5, 2], [300, 129], 8, 2, 128, extra=5)
    o1, l1 = run_oracle(wl)
    rng = np.random.default_rng(0)
    perm = rng.permutation(wl.num_pages)            # new physical position of each page
    pool2 = torch.empty_like(wl.kv_pool)
    pool2[torch.from_numpy(perm)] = wl.kv_pool
    bt = wl.block_table.numpy().copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    wl.kv_pool, wl.block_table = pool2, torch.from_numpy(bt)
    o2, l2 = run_oracle(wl)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_thread_count_and_row_subset_are_bitwise():
    wl = small(10, [7, 3], [100, 64], 6, 3, 128)
    o1, l1 = run_oracle(wl, n_threads=1)
    o2, l2 = run_oracle(wl, n_threads=7)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    rows = [9, 0, 4]
    o3, l3 = run_oracle(wl, rows=rows)
    assert np.array_equal(o3, o1[rows]) and np.array_equal(l3, l1[rows])


def test_key_offset_invariance():
    # Adding one vector c to every K row of a (sequence, kv head) adds q.c to every
    # score of a query row, which softmax ignores. K and c are chosen so that
    # K + c stays exact in bf16.
    wl = small(11, [4, 2], [90, 33], 4, 2, 16, causal=True)
    rng = np.random.default_rng(1)
    live = wl.kv_pool.float().isfinite()
    k = torch.from_numpy(rng.integers(-8, 9, size=wl.kv_pool[:, 0].shape).astype(np.float32) / 4)
    wl.kv_pool[:, 0] = torch.where(live[:, 0], k, wl.kv_pool[:, 0].float()).to(torch.bfloat16)
    o1, _ = run_oracle(wl)
    c = torch.from_numpy(rng.integers(-8, 9, size=(2, 16)).astype(np.float32))
    wl.kv_pool[:, 0] = (wl.kv_pool[:, 0].float() + c[None, None]).to(torch.bfloat16)
    assert torch.equal(wl.kv_pool[:, 0].float()[live[:, 0]],
                       (k + c[None, None]).expand_as(live[:, 0])[live[:, 0]])
    o2, _ = run_oracle(wl)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-10)


def test_gqa_equals_mha_with_repeated_heads():
    g = 3
    wl = small(12, [3, 4], [70, 140], 6, 2, 128)
    o1, l1 = run_oracle(wl)
    pool = wl.kv_pool.repeat_interleave(g, dim=3).contiguous()
    o2, l2 = oracle.forward(wl.q, pool, wl.block_table, wl.seq_lens, wl.cu_q, 6, 6, 128, 64,
                            wl.scale, wl.causal)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_split_identity_with_combine():
    wl = small(13, [3, 1, 6], [500, 257, 64], 4, 2, 128)
    full_o, full_l = run_oracle(wl)
    for cuts in ([0, 100, 300, -1], [0, 64, 65, 128, 129, 640, -1], [0, 1, -1]):
        parts_o, parts_l = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            o, l = run_oracle(wl, key_window=(a, b))
            parts_o.append(o.reshape(-1, 128))
            parts_l.append(l.reshape(-1))
        co, cl = oracle.combine(np.stack(parts_o), np.stack(parts_l))
        np.testing.assert_allclose(co, full_o.reshape(-1, 128), rtol=0, atol=1e-12)
        np.testing.assert_allclose(cl, full_l.reshape(-1), rtol=0, atol=1e-12)


def test_combine_of_empty_parts():
    co, cl = oracle.combine(np.zeros((2, 1, 4)), np.full((2, 1), -np.inf))
    assert np.all(co == 0) and np.isneginf(cl[0])
    vals = np.arange(4.0)[None, None]
    co, cl = oracle.combine(np.concatenate([vals, np.ones((1, 1, 4)) * 7]), np.array([[0.5], [-np.inf]]))
    assert np.array_equal(co[0], np.arange(4.0)) and cl[0] == 0.5


def test_contiguous_equals_identity_paged():
    wl = workloads.make_contiguous("c", 14, [5, 2], [130, 64], 4, 2, 128, causal=True)
    o1, l1 = run_oracle(wl)
    # lay the same rows out as pages of 64 with an identity-like table
    P, H, D = 64, 2, 128
    kv = wl.kv_pool
    pages, table = [], []
    start = 0
    for L in wl.seq_lens.tolist():
        row = []
        for s in range((L + P - 1) // P):
            blk = torch.full((2, P, H, D), float("nan"), dtype=torch.bfloat16)
            n = min(P, L - s * P)
            blk[:, :n] = kv[:, start + s * P:start + s * P + n]
            row.append(len(pages))
            pages.append(blk)
        start += L
        table.append(row)
    width = max(len(r) for r in table)
    bt = torch.tensor([r + [-1] * (width - len(r)) for r in table], dtype=torch.int32)
    pool = torch.stack(pages)
    o2, l2 = oracle.forward(wl.q, pool, bt, wl.seq_lens, wl.cu_q, 4, 2, 128, 64, wl.scale, True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_interleaved_manifest_layout_matches_split_layout():
    """The decode manifest's 6-D kv buffer interleaves K and V per head; same result."""
    wl = small(15, [8, 8], [300, 650], 24, 4, 256, extra=6)
    o1, l1 = run_oracle(wl)
    n, _, P, H, D = wl.kv_pool.shape
    pool6 = torch.full((n, 2, P, H, 2, D), float("nan"), dtype=torch.bfloat16)
    pool6[:, 0, :, :, 0] = wl.kv_pool[:, 0]
    pool6[:, 0, :, :, 1] = wl.kv_pool[:, 1]
    st = oracle.pool_strides(H, D, P, "paged_interleaved")
    o2, l2 = oracle.forward(wl.q, pool6, wl.block_table, wl.seq_lens, wl.cu_q, 24, 4, 256, 64,
                            wl.scale, True, strides=st)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_nan_outside_live_rows_never_reaches_the_output():
    wl = workloads.named(1)
    assert torch.isnan(wl.kv_pool.float()).any()
    o, l = run_oracle(wl)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    ro, rl = dense_attention(wl)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# constants printed by the decode manifest (tests/golden)
# ----------------------------------------------------------------------------
def _golden():
    with open(os.path.join(HERE, "golden", "decode_manifest_constants.json")) as f:
        return json.load(f)


def test_manifest_scale_is_scale_times_log2e():
    g = _golden()["pack_scalars"]
    c = np.float32(1.0 / 16) * np.float32(math.log2(math.e))
    assert int(np.array([c], np.float32).view(np.int32)[0]) == g["softmax_scale_log2e_at_1220_i32"]


def test_manifest_head_grouping_is_contiguous():
    g = _golden()
    ps = g["pack_scalars"]
    magic = ps["divmod_magic_at_1180_i32"] & 0xFFFFFFFF
    shift = 32 + ps["divmod_shift_at_1188"]
    G = ps["group_at_1172"]
    assert ps["n_heads_q_at_1168"] == G * ps["n_heads_kv_at_1164"]
    for h in range(ps["n_heads_q_at_1168"]):
        assert (h * magic) >> shift == h // G
    # Q tensor map: dims [D, group, kv head, token], group innermost after D
    qt = g["q_tensormap"]
    D, Gd, H, _ = qt["dims"]
    assert qt["strides_bytes"] == [D * 2, D * 2 * Gd, D * 2 * Gd * H]
    assert ps["q_token_stride_at_1192"] == D * Gd * H
    # and the oracle maps q head h to kv head h // G: with KV heads that differ,
    # each q head's output must equal the MHA output of its own kv head
    wl = small(16, [2], [40], 6, 2, 16)
    o, _ = run_oracle(wl)
    pool = wl.kv_pool.repeat_interleave(3, dim=3).contiguous()
    o2, _ = oracle.forward(wl.q, pool, wl.block_table, wl.seq_lens, wl.cu_q, 6, 6, 16, 64, wl.scale, True)
    assert np.array_equal(o, o2)


def test_manifest_cache_strides_and_table_width():
    g = _golden()
    kt = g["k_tensormap"]
    D, H, P = 256, 4, 64
    s_page, s_kv, s_row, s_head = oracle.pool_strides(H, D, P, "paged_interleaved")
    assert [s_row * 2, s_head * 2, s_page * 2] == [kt["row_stride_bytes"], kt["head_stride_bytes"],
                                                     kt["page_stride_bytes"]]
    off = g["program_kv_offsets"]
    assert off["v_offset_bytes"] - off["k_offset_bytes"] == s_kv * 2
    lens = g["kv_lengths_of_the_example"]["kv_lens"]
    width = max((L + P - 1) // P for L in lens)
    assert g["buffers"]["table_shape"] == [2, width]
    assert g["pack_scalars"]["per_seq_capacity_at_1148"] == width * P
    assert g["pack_scalars"]["max_pages_per_seq_at_1160"] == width
    wl = workloads.named(1)
    assert list(wl.block_table.shape) == g["buffers"]["table_shape"]
    assert wl.num_pages == g["buffers"]["kv_shape"][0]
