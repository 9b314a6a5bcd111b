"""GPU parity of pattn_forward_append: the cache write of the new tokens' K and V
rows (the GB10 graph's kv_write node) followed by attention over the updated
cache, against the oracle's write on a copy of the pool and its attention.

The pool after the call must equal the oracle's pool bit for bit (NaN pages
included); the output must meet the parity bar against the float64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_parity, sample_rows, to_device

pytestmark = pytest.mark.gpu


def run_append(wl, d, k, v, check=True):
    import paged_kv_flashattention_varlen_gb300 as pk
    out = torch.full_like(d["q"], float("nan"))
    kd, vd = k.to(d["q"].device), v.to(d["q"].device)
    rc = pk.forward_append(out, d["q"], kd, vd, d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q,
                           max_kv=wl.max_kv, n_heads_kv=wl.n_heads_kv, scale=wl.scale,
                           causal=wl.causal, num_pages=wl.num_pages, check=check)
    torch.cuda.synchronize()
    return out, rc


def _same_bits(a, b):
    return torch.equal(a.cpu().view(torch.int16), b.cpu().view(torch.int16))


@pytest.mark.parametrize("index,scale_down,all_rows", [
    (1, 1, True),    # tiny paged decode, 8 new tokens per sequence, D 256
    (2, 1, True),    # decode batch, one new token per sequence
    (3, 16, True),   # causal prefill 4 x 512: every token is new
    (4, 32, True),   # contiguous cache, non-causal
    (5, 4, False),   # mixed decode + chunks, D 256
])
def test_append_then_attend(index, scale_down, all_rows):
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = workloads.named(index, scale_down=scale_down)
    k, v = workloads.new_kv_rows(wl, 500 + index)
    ref_wl = oracle.append_workload(wl, k, v)
    d = to_device(wl)
    out, _ = run_append(wl, d, k, v)
    assert pk.device_status() == 0
    assert _same_bits(d["kv"], ref_wl.kv_pool), "cache after the write differs from the oracle's"
    rows = None if all_rows else sample_rows(ref_wl, per_seq=4)
    assert_parity(out, ref_wl, rows=rows)


def test_append_equals_write_then_forward():
    """The attention of the append call is the plain forward over the written cache."""
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = workloads.named(2, scale_down=4)
    k, v = workloads.new_kv_rows(wl, 77)
    d = to_device(wl)
    out_a, _ = run_append(wl, d, k, v)
    out_f = torch.full_like(out_a, float("nan"))
    pk.forward(out_f, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q, max_kv=wl.max_kv,
               n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal, num_pages=wl.num_pages)
    torch.cuda.synchronize()
    assert _same_bits(out_a, out_f)


def test_more_queries_than_keys_writes_only_slotted_tokens():
    # sequence 1 has ql = 6 > L = 4 (non-causal so that its rows attend): tokens
    # 0 and 1 of it have no cache slot and are not written
    wl = workloads.make_paged("q_gt_l", 31, [2, 6], [100, 4], 8, 2, 128, causal=False, extra_pages=2)
    k, v = workloads.new_kv_rows(wl, 9)
    ref_wl = oracle.append_workload(wl, k, v)
    d = to_device(wl)
    out, _ = run_append(wl, d, k, v)
    assert _same_bits(d["kv"], ref_wl.kv_pool)
    assert_parity(out, ref_wl)


def test_bad_page_in_the_new_rows_is_rejected_without_writing():
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = workloads.make_paged("badpage", 41, [3, 3], [70, 130], 8, 2, 128, causal=True, extra_pages=2)
    k, v = workloads.new_kv_rows(wl, 10)
    bt = wl.block_table.clone()
    bt[1, (130 - 1) // 64] = wl.num_pages + 5  # the slot of sequence 1's new tokens
    bad = workloads.Workload(**{**wl.__dict__, "block_table": bt})
    d = to_device(bad)
    pool_before = d["kv"].clone()
    out, rc = run_append(bad, d, k, v, check=False)
    assert rc == 0
    assert pk.device_status() == 5
    # sequence 0 written and attended as usual; sequence 1 untouched and zero
    ref_wl = oracle.append_workload(wl, k, v)
    cu = wl.cu_q.tolist()
    pages0 = wl.block_table[0, :2].tolist()
    for pg in pages0:
        assert _same_bits(d["kv"][pg], ref_wl.kv_pool[pg])
    others = [p for p in range(wl.num_pages) if p not in pages0]
    assert _same_bits(d["kv"][others], pool_before[others])
    assert torch.count_nonzero(out[cu[1]:cu[2]].float()) == 0
    ref0, _ = oracle.forward_workload(ref_wl, rows=list(range(cu[0], cu[1])))
    got0 = out[cu[0]:cu[1]].float().cpu().numpy()
    assert np.abs(got0 - ref0).max() <= 2e-2
