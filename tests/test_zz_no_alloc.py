"""pattn_forward_noalloc: attention without any device allocation.

Some callers cannot let a library call cudaMalloc: a serving process whose
caching allocator already holds nearly all of the GPU, a decode loop that
cannot afford the device synchronisation an allocation implies, a host that
owns every device buffer itself. For them the library has one more entry
point that works from a fixed device array compiled into the library. These
tests call it through the C ABI, twice in a row (the array keeps the previous
call's contents), and check each output element by element against the
float64 oracle and against pattn_forward, within the parity bar of the other
tests. They also check that a batch too large for the array is refused before
anything runs, and that a rejected page behind this entry point is reported by
pattn_get_device_status.

This file is collected last, so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads
from helpers import MAX_ABS, MEAN_ABS, assert_parity, run_gpu, to_device

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.fixture(scope="module")
def lib():
    from paged_kv_flashattention_varlen_gb300 import _lib, build
    build.build()
    return _lib.load()


def _noalloc(lib, wl, d, out):
    bt = d["bt"]
    return lib.pattn_forward_noalloc(
        out.data_ptr(), d["q"].data_ptr(), d["kv"].data_ptr(),
        None if bt is None else bt.data_ptr(), d["sl"].data_ptr(), d["cu"].data_ptr(),
        wl.num_seqs, wl.total_q, wl.max_q, wl.max_kv, wl.n_heads_q, wl.n_heads_kv, wl.head_dim,
        wl.page_size, wl.num_pages, float(wl.scale), int(wl.causal),
        torch.cuda.current_stream().cuda_stream)


def _decode_d256():
    # decode sequences of the hybrid model's full-attention layer (16/2 heads, D 256),
    # one or two query tokens each
    rng = np.random.default_rng(5)
    kv = rng.integers(200, 2000, size=32).tolist()
    return workloads.make_paged("noalloc_d256", 77, [1, 2] * 16, kv, 16, 2, 256, 64,
                                scale=1.0 / 16, causal=True)


def _split_decode_and_prefill():
    # 16/2 heads (G 8), D 128, every sequence at 32768 keys: two-token sequences
    # (16 packed rows) are decode units, four-token ones (32 rows, one q tile)
    # single-tile prefill units, and both kinds split their KV range, each list
    # sized from its own work, so the batch needs about twice one list's splits
    return workloads.make_paged("noalloc_splits", 78, [4, 2] * 5, [32768] * 10, 16, 2, 128, 64,
                                causal=True)


CASES = {"tiny_decode": lambda: workloads.named(1),
         "decode_batch": lambda: workloads.named(2, scale_down=4),
         "decode_d256": _decode_d256,
         "split_decode_and_prefill": _split_decode_and_prefill}


@pytest.mark.parametrize("which", list(CASES))
def test_noalloc_matches_oracle_and_forward_two_calls_in_a_row(lib, which):
    wl = CASES[which]()
    d = to_device(wl)
    ref = run_gpu(wl, d=d).float()
    for _ in range(2):
        out = torch.full_like(d["q"], float("nan"))
        rc = _noalloc(lib, wl, d, out)
        assert rc == 0, lib.pattn_status_string(rc)
        assert lib.pattn_get_device_status(torch.cuda.current_stream().cuda_stream) == 0
        assert_parity(out, wl)
        diff = (out.float() - ref).abs()
        assert diff.max().item() <= MAX_ABS and diff.mean().item() <= MEAN_ABS


def test_noalloc_split_case_needs_more_than_one_list_of_splits(lib):
    # the batch above really needs more partial rows than "one item target plus
    # the units" would give: the scratch bound must count both lists
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = _split_decode_and_prefill()
    d = to_device(wl)
    _, _, counts = pk.plan_items(d["bt"], d["sl"], d["cu"], total_q=wl.total_q, max_q=wl.max_q,
                                 max_kv=wl.max_kv, n_heads_q=wl.n_heads_q, n_heads_kv=wl.n_heads_kv,
                                 head_dim=wl.head_dim, causal=wl.causal, num_pages=wl.num_pages)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    target = min(4 * sms // 2, 512)
    units = wl.num_seqs * wl.n_heads_kv
    rows_cap = min(128, wl.max_q * wl.n_heads_q // wl.n_heads_kv)
    assert counts[3] > (target + units) * rows_cap


def test_noalloc_bad_page_is_reported_and_its_rows_zeroed(lib):
    wl = workloads.make_paged("noalloc_bad", 79, [2, 2, 1], [100, 100, 700], 8, 2, 128, 64, causal=True)
    d = to_device(wl)
    bt = d["bt"].clone()
    bt[1, 1] = wl.num_pages + 5
    d["bt"] = bt
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.pattn_get_device_status(stream) == 0
    out = torch.full_like(d["q"], float("nan"))
    assert _noalloc(lib, wl, d, out) == 0
    assert lib.pattn_get_device_status(stream) == 5  # PATTN_ERR_DEVICE_BAD_INPUT
    assert lib.pattn_get_device_status(stream) == 0  # read and cleared
    assert torch.all(out[2:4] == 0)
    assert_parity(out, wl, rows=[0, 1, 4])


def test_noalloc_refuses_a_batch_beyond_its_scratch(lib):
    # 4096 single-token sequences over 8 KV heads need far more than the scratch holds
    B, hq, hkv, D = 4096, 32, 8, 128
    need = lib.pattn_workspace_size(B, B, 1, 64, hq, hkv, D, 64)
    assert need > (16 << 20)
    dev = torch.device("cuda:0")
    q = torch.zeros(B, hq, D, dtype=torch.bfloat16, device=dev)
    out = torch.full_like(q, 7.0)
    kv = torch.zeros(B, 2, 64, hkv, D, dtype=torch.bfloat16, device=dev)
    bt = torch.arange(B, dtype=torch.int32, device=dev).view(B, 1)
    sl = torch.ones(B, dtype=torch.int32, device=dev)
    cu = torch.arange(B + 1, dtype=torch.int32, device=dev)
    rc = lib.pattn_forward_noalloc(out.data_ptr(), q.data_ptr(), kv.data_ptr(), bt.data_ptr(),
                                   sl.data_ptr(), cu.data_ptr(), B, B, 1, 64, hq, hkv, D, 64, B,
                                   0.1, 1, torch.cuda.current_stream().cuda_stream)
    assert rc == 4  # PATTN_ERR_NO_MEMORY: refused before any launch
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
