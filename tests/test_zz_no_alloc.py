"""pattn_forward_noalloc: attention without any device allocation.

Some callers cannot let a library call cudaMalloc: a serving process whose
caching allocator already holds nearly all of the GPU, a decode loop that
cannot afford the device synchronisation an allocation implies, a host that
owns every device buffer itself. For them the library has one more entry
point that works from a fixed device array compiled into the library. These
tests call it through the C ABI and check it against pattn_forward, twice in a
row (the array keeps the previous call's contents), and check that a batch
too large for the array is refused before anything runs.

This file is collected last, so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads
from helpers import MAX_ABS, MEAN_ABS, run_gpu, to_device

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


@pytest.mark.parametrize("which", ["tiny_decode", "decode_batch", "decode_d256"])
def test_noalloc_matches_forward_two_calls_in_a_row(lib, which):
    wl = {"tiny_decode": lambda: workloads.named(1),
          "decode_batch": lambda: workloads.named(2, scale_down=4),
          "decode_d256": _decode_d256}[which]()
    d = to_device(wl)
    ref = run_gpu(wl, d=d).float()
    for _ in range(2):
        out = torch.full_like(d["q"], float("nan"))
        rc = _noalloc(lib, wl, d, out)
        assert rc == 0, lib.pattn_status_string(rc)
        torch.cuda.synchronize()
        got = out.float()
        assert torch.isfinite(got).all()
        diff = (got - ref).abs()
        assert diff.max().item() <= MAX_ABS and diff.mean().item() <= MEAN_ABS


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
