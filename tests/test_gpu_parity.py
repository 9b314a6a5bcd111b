"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small cases are compared element by element over every output; the five named
workloads at full size are compared over every decode row and over sampled
prefill rows, which the oracle computes one by one: the first and last rows of
each sequence, the rows on both sides of every q-tile boundary (so that every
q tile, and with all heads every work item of the persistent schedule, has
checked rows) and seeded random rows, at least 1024 query rows x all heads per
prefill workload. Bar: max |err| <= 2e-2 and mean |err| <= 2e-3 on the bf16
outputs.
"""
import numpy as np
import pytest
import torch

import workloads
from helpers import assert_parity, run_gpu, sample_rows, to_device

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_flashattention_varlen_gb300 import build
    build.build()
    import paged_kv_flashattention_varlen_gb300 as pk
    assert pk.device_status() == 0


def _status():
    import paged_kv_flashattention_varlen_gb300 as pk
    return pk.device_status()


# --------------------------------------------------------------- named workloads
def test_tiny_paged_decode_full():
    wl = workloads.named(1)
    out = run_gpu(wl)
    assert_parity(out, wl)
    assert _status() == 0


def test_decode_batch_full():
    wl = workloads.named(2)
    out = run_gpu(wl)
    assert_parity(out, wl)
    assert _status() == 0


def test_causal_prefill_small_full():
    wl = workloads.named(3, scale_down=16)      # 4 x 512 tokens, every row
    out = run_gpu(wl)
    assert_parity(out, wl)


def test_causal_prefill_full_size_every_tile_boundary_over_3000_rows():
    # 4 x 8192 tokens in q tiles of 32 tokens (G 4): rows q0-1, q0, q0+1 at each
    # of the 255 boundaries per sequence, first/last and random rows
    wl = workloads.named(3)
    out = run_gpu(wl)
    rows = sample_rows(wl, per_seq=8, every_boundary=True, min_rows=1024)
    assert len(rows) >= 3000
    assert_parity(out, wl, rows=rows)
    assert _status() == 0


def test_noncausal_contiguous_small_full():
    wl = workloads.named(4, scale_down=32)      # 1181 tokens, every row
    out = run_gpu(wl)
    assert_parity(out, wl)


def test_noncausal_contiguous_full_size_every_tile_boundary_1024_rows():
    # 37,810 tokens in q tiles of 128 (G 1): rows q0-1, q0, q0+1 at each of the
    # 295 boundaries, first/last rows, random rows up to 1024 rows x 56 heads
    wl = workloads.named(4)
    out = run_gpu(wl)
    rows = sample_rows(wl, per_seq=4, every_boundary=True, min_rows=1024)
    assert len(rows) >= 1024
    assert_parity(out, wl, rows=rows)
    assert _status() == 0


@pytest.mark.parametrize("n", [37760, 37761])
def test_noncausal_tail_lengths_every_tile_boundary(n):
    # the video-DiT page's tail study: the 37,810-token shape cut to a multiple
    # of the 128-row tile (37,760 = 295 x 128) and one past it, same recipe as
    # the named workload (56 heads MHA, contiguous cache, K channel offsets);
    # rows on both sides of every q-tile boundary and the last tile's rows
    wl = workloads.make_contiguous("tail", workloads.seed_for(4) + n, [n], [n], 56, 56, 128,
                                   scale=1.0 / np.sqrt(128), causal=False, k_offset_std=0.5)
    out = run_gpu(wl)
    rows = sorted(set(sample_rows(wl, per_seq=4, every_boundary=True)) | {n - 129, n - 128, n - 2, n - 1})
    assert len(rows) >= 3 * (n // 128)
    assert_parity(out, wl, rows=rows)
    assert _status() == 0


def test_mixed_batch_small_full():
    wl = workloads.named(5, scale_down=8)
    out = run_gpu(wl)
    assert_parity(out, wl)


def test_mixed_batch_full_size_every_decode_row_and_chunk_tile_boundary():
    # all 96 decode rows; the four 2048-token chunks in q tiles of 16 tokens
    # (G 8; pairs of q tiles on the CTA-pair kernel): rows on both sides of
    # every boundary, first/last and random rows, over 1500 chunk rows
    wl = workloads.named(5)
    out = run_gpu(wl)
    decode_rows = list(range(96))
    assert_parity(out, wl, rows=decode_rows)
    chunk_rows = [r for r in sample_rows(wl, per_seq=6, every_boundary=True, min_rows=1024) if r >= 96]
    assert len(chunk_rows) >= 1500
    assert_parity(out, wl, rows=chunk_rows)
    assert _status() == 0


# --------------------------------------------------------------- edge sweep
EDGES = [1, 63, 64, 65, 127, 128, 129]


@pytest.mark.parametrize("d,hq,hkv", [(128, 4, 1), (128, 8, 8), (256, 12, 2), (256, 16, 2)])
@pytest.mark.parametrize("causal", [True, False])
def test_edge_lengths(d, hq, hkv, causal):
    kv_lens, q_lens = [], []
    for L in EDGES:
        for ql in EDGES:
            if causal and ql > L:
                continue
            kv_lens.append(L)
            q_lens.append(ql)
    wl = workloads.make_paged("edges", 500 + d + hq, q_lens, kv_lens, hq, hkv, d, 64,
                              causal=causal, extra_pages=3)
    out = run_gpu(wl)
    assert_parity(out, wl)
    assert _status() == 0


@pytest.mark.parametrize("hq,hkv", [(6, 1), (7, 1), (16, 1), (32, 2)])
@pytest.mark.parametrize("causal", [True, False])
def test_head_dim_128_group_sizes_full_and_partial_q_tiles(hq, hkv, causal):
    # head_dim 128 prefill at G = 6, 7, 16, 32 (q tiles of 21, 18, 8 and 4
    # tokens: 126, 126, 128 and 128 rows). Full q tiles of unsplit items leave
    # through the tensor store of [32, G, 1, T] boxes; the last, partial q tile
    # of each sequence and the split single-q-tile units store row by row.
    g = hq // hkv
    t = 128 // g
    q_lens = [3 * t, 3 * t + 1, t - 1, 200, 1, 2 * t]
    kv_lens = [3 * t, 700, 9000, 1300, 64, 4 * t + 5]
    wl = workloads.make_paged("groups128", 610 + hq + int(causal), q_lens, kv_lens, hq, hkv, 128, 64,
                              causal=causal, extra_pages=2)
    out = run_gpu(wl)
    assert_parity(out, wl)
    assert _status() == 0


def test_long_decode_splits_and_short_sequences_mixed():
    rng = np.random.default_rng(7)
    kv = [1, 2, 64, 65, 129, 4000, 20000, 300, 8191, 8192, 8193]
    wl = workloads.make_paged("splits", 8, [1] * len(kv), kv, 32, 8, 128, 64, causal=True,
                              extra_pages=2)
    out = run_gpu(wl)
    assert_parity(out, wl)
    wl2 = workloads.make_paged("splits256", 9, [1, 3, 1] * 4, rng.integers(1, 9000, size=12),
                               16, 2, 256, 64, causal=True)
    assert_parity(run_gpu(wl2), wl2)


@pytest.mark.parametrize("causal", [True, False])
def test_head_dim_256_pairs_with_single_tile_and_split_units(causal):
    # head_dim 256, G 8 (16 tokens per q tile): the CTA-pair kernel takes items
    # of two q tiles; a 40-token sequence ends in a half pair, 3- and 2-token
    # sequences (one q tile, long KV ranges) run as split items with the pair's
    # second CTA holding no rows, and 1-token sequences go to the decode kernel
    q_lens = [3, 40, 1, 17, 33, 2, 130]
    kv_lens = [6000, 300, 5000, 17, 2000, 65, 8191]
    wl = workloads.make_paged("pairs256", 21 + causal, q_lens, kv_lens, 16, 2, 256, 64,
                              causal=causal, extra_pages=3)
    assert_parity(run_gpu(wl), wl)
    assert _status() == 0


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 2)])
def test_head_dim_256_pairs_group_sizes(hq, hkv):
    # G 1 (128 tokens per q tile, pairs of 256 tokens) and G 16 (8 tokens per
    # q tile): ragged lengths, a half pair at each sequence end
    wl = workloads.make_paged("pairsg", 24 + hq, [300, 9, 130, 1], [300, 520, 4000, 77], hq, hkv, 256, 64,
                              causal=True, extra_pages=2)
    assert_parity(run_gpu(wl), wl)
    assert _status() == 0


def test_head_dim_256_contiguous_pairs():
    wl = workloads.make_contiguous("pairs256c", 23, [37, 200, 5], [37, 900, 5], 32, 4, 256,
                                   causal=True)
    assert_parity(run_gpu(wl), wl)
    assert _status() == 0


# --------------------------------------------------------------- degenerate inputs
def test_empty_and_queries_before_the_first_key():
    # L = 0 (no key), ql = 0 (no query), and non-causal/causal ql > L rows
    wl = workloads.make_paged("empty", 11, [3, 0, 5, 2], [0, 10, 3, 70], 8, 2, 128, 64,
                              causal=True, extra_pages=1)
    out = run_gpu(wl)
    assert_parity(out, wl)
    assert torch.all(out[:3] == 0)
    assert torch.all(out[3:5] == 0)   # positions 3-5+i < 0 for i < 2
    assert _status() == 0


def test_bad_page_sets_error_and_zeroes_that_sequence():
    wl = workloads.make_paged("bad", 12, [2, 2], [100, 100], 8, 2, 128, 64, causal=True)
    d = to_device(wl)
    bt = d["bt"].clone()
    bt[1, 1] = wl.num_pages + 5
    d["bt"] = bt
    out = run_gpu(wl, d=d)
    import paged_kv_flashattention_varlen_gb300 as pk
    assert pk.device_status() == 5
    assert torch.all(out[2:4] == 0)
    assert_parity(out, wl, rows=[0, 1])
    assert pk.device_status() == 0


def test_lengths_beyond_host_bounds_are_rejected_on_device():
    wl = workloads.make_paged("bounds", 13, [2, 1], [100, 50], 8, 2, 128, 64, causal=True)
    d = to_device(wl)
    d["bt"] = d["bt"][:, :1].contiguous()           # table stride ceil(max_kv / 64) = 1
    import paged_kv_flashattention_varlen_gb300 as pk
    out = torch.full_like(d["q"], float("nan"))
    pk.forward(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=2, max_kv=64,
               n_heads_kv=2, scale=wl.scale, causal=True, num_pages=wl.num_pages)
    assert pk.device_status() == 5
    assert torch.all(out[:2] == 0)                  # L = 100 > max_kv: rejected
    assert_parity(out, wl, rows=[2])


@pytest.mark.parametrize("d,hq,hkv", [(256, 24, 4), (128, 8, 2)])
def test_decode_sized_sequence_that_the_bounds_rule_out_runs_on_the_prefill_kernel(d, hq, hkv):
    # The decode kernel is not launched when every sequence must hold more than
    # 16 / G queries (total_q - (B - 1) * max_q of them). A caller whose cu_q
    # ends short of total_q can still pass a sequence of one query: the plan
    # then gives its unit to the prefill kernel, which serves it exactly.
    wl = workloads.make_paged("short_seq", 15, [1, 8, 3], [300, 650, 129], hq, hkv, d, 64, causal=True)
    d_in = to_device(wl)
    pad = 40  # rows past cu_q[B]: total_q - 2 * max_q > 16 / G
    d_in["q"] = torch.cat([d_in["q"], torch.randn(pad, hq, d, device="cuda").to(torch.bfloat16)])
    import paged_kv_flashattention_varlen_gb300 as pk
    pre, dec, _ = pk.plan_items(d_in["bt"], d_in["sl"], d_in["cu"], total_q=wl.total_q + pad,
                                max_q=wl.max_q, max_kv=wl.max_kv, n_heads_q=hq, n_heads_kv=hkv,
                                head_dim=d, causal=True, num_pages=wl.num_pages)
    assert dec.shape[0] == 0 and (pre[:, 0] & 0xFFFFFF == 0).any()  # sequence 0 on the prefill list
    out = torch.full_like(d_in["q"], float("nan"))
    run_gpu(wl, d=d_in, out=out)
    assert_parity(out[:wl.total_q], wl)
    assert torch.isnan(out[wl.total_q:].float()).all()  # rows of no sequence are not written
    assert _status() == 0


# --------------------------------------------------------------- invariants on the GPU
def test_repeatable_and_page_permutation_bitwise():
    wl = workloads.named(2, scale_down=4)
    d = to_device(wl)
    a = run_gpu(wl, d=d)
    b = run_gpu(wl, d=d)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    perm = torch.from_numpy(np.random.default_rng(3).permutation(wl.num_pages))
    pool2 = torch.empty_like(wl.kv_pool)
    pool2[perm] = wl.kv_pool
    bt = wl.block_table.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    d2 = dict(d, kv=pool2.cuda(), bt=bt.cuda())
    c = run_gpu(wl, d=d2)
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_contiguous_equals_paged_bitwise():
    wl = workloads.make_contiguous("c", 14, [40, 1, 7], [300, 129, 64], 8, 2, 128, causal=True)
    a = run_gpu(wl)
    # same rows laid out as pages of 64
    P = 64
    pages, table, start = [], [], 0
    for L in wl.seq_lens.tolist():
        row = []
        for s in range((L + P - 1) // P):
            blk = torch.full((2, P, 2, 128), float("nan"), dtype=torch.bfloat16)
            n = min(P, L - s * P)
            blk[:, :n] = wl.kv_pool[:, start + s * P:start + s * P + n]
            row.append(len(pages))
            pages.append(blk)
        start += L
        table.append(row)
    w = max(len(r) for r in table)
    wl.block_table = torch.tensor([r + [-1] * (w - len(r)) for r in table], dtype=torch.int32)
    wl.kv_pool = torch.stack(pages)
    wl.num_pages = len(pages)
    b = run_gpu(wl)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_host_entry_point_matches_device_entry_point():
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = workloads.named(1)
    a = run_gpu(wl)
    out = torch.empty_like(wl.q).pin_memory()
    pk.forward_host(out, wl.q.pin_memory(), wl.kv_pool.pin_memory(), wl.block_table.pin_memory(),
                    wl.seq_lens, wl.cu_q, max_q=wl.max_q, max_kv=wl.max_kv,
                    n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                    num_pages=wl.num_pages)
    assert torch.equal(a.cpu().view(torch.int16), out.view(torch.int16))


def test_profile_counts_launches():
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = workloads.named(1)
    d = to_device(wl)
    pk.profile_read()
    pk.profile_enable(True)
    for _ in range(3):
        run_gpu(wl, d=d)
    pk.profile_enable(False)
    plan, attn, comb, calls = pk.profile_read()
    assert calls == 3 and attn > 0 and plan > 0


# --------------------------------------------------------------- failure detection
def test_bounded_wait_runs_out_into_an_error_status_and_the_context_survives():
    # a wait on an mbarrier phase that nothing completes gives up after its
    # limit, sets the timeout bit and returns: the host reads the status, and
    # the next call on the same context runs normally
    import paged_kv_flashattention_varlen_gb300 as pk
    pk.selftest_wait_timeout()
    assert pk.device_status() == 6  # PATTN_ERR_DEVICE_TIMEOUT
    assert pk.device_status() == 0  # read and cleared
    wl = workloads.named(2, scale_down=8)
    assert_parity(run_gpu(wl), wl)
    assert _status() == 0


@pytest.mark.parametrize("which", ["decode", "prefill", "prefill_two_q"])
def test_attention_kernel_abort_path_reports_timeout_and_the_context_survives(which):
    # the first CTA's MMA-issuing thread of the decode kernel (a decode batch),
    # of the one-q-tile prefill kernel (a causal prefill batch) or of the
    # two-q-tile prefill kernel (a non-causal batch) waits on a phase that
    # nothing completes: after the wait limit every role of that CTA leaves its
    # loop, drains its in-flight copies and MMAs and frees its tensor memory;
    # the host reads the timeout, and the next ordinary call on the same
    # context passes parity
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = {"decode": lambda: workloads.named(2, scale_down=8),
          "prefill": lambda: workloads.named(3, scale_down=16),
          "prefill_two_q": lambda: workloads.named(4, scale_down=32)}[which]()
    d = to_device(wl)
    out = torch.full_like(d["q"], float("nan"))
    pk.selftest_attention_timeout(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q,
                                  max_kv=wl.max_kv, n_heads_kv=wl.n_heads_kv, scale=wl.scale,
                                  causal=wl.causal, num_pages=wl.num_pages)
    assert pk.device_status() == 6  # PATTN_ERR_DEVICE_TIMEOUT
    assert pk.device_status() == 0
    assert_parity(run_gpu(wl, d=d), wl)
    assert _status() == 0


@pytest.mark.parametrize("world", [2, 4])
def test_head_shards_through_the_library_reassemble_the_output(world):
    # head (tensor) sharding as one process per GPU would run it, one shard
    # after the other on this GPU: each shard's KV heads and query heads through
    # the C ABI, the blocks concatenated along the heads against the oracle
    import paged_kv_flashattention_varlen_gb300 as pk
    from paged_kv_flashattention_varlen_gb300 import dist as pdist
    wl = workloads.make_paged("heads_gpu", 18, [1, 40, 300, 2], [700, 200, 900, 5000], 32, 8, 128, 64,
                              causal=True, extra_pages=2)
    blocks = []
    for r in range(world):
        q_r, kv_r, hq_r, hkv_r = pdist.shard_heads(wl.q, wl.kv_pool, wl.n_heads_q, wl.n_heads_kv, world, r)
        part = workloads.Workload(**{**wl.__dict__, "q": q_r, "kv_pool": kv_r, "n_heads_q": hq_r,
                                     "n_heads_kv": hkv_r})
        blocks.append(run_gpu(part))
        assert _status() == 0
    assert_parity(torch.cat(blocks, dim=1), wl)
