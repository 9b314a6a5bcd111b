"""GPU parity on seeded random shapes: batch sizes, query and KV lengths, head
groups, head dims, causal or not, paged or contiguous, each case compared with
the float64 oracle over every output row. The shapes mix decode units (at most
16 packed query rows, on the swap-AB kernel), prefill units, split units and partial q tiles in one
call, so that both attention kernels, the planner's split rule and the two
output paths of the prefill kernel meet in the same launch."""
import numpy as np
import pytest
import torch

import workloads
from helpers import assert_parity, run_gpu, to_device

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_flashattention_varlen_gb300 import build
    build.build()


GROUPS = {128: [(4, 1), (8, 2), (12, 2), (32, 8), (5, 5), (16, 1)],
          256: [(8, 1), (16, 2), (24, 4), (4, 4)]}


def _case(seed):
    rng = np.random.default_rng(seed)
    d = int(rng.choice([128, 256]))
    hq, hkv = GROUPS[d][int(rng.integers(len(GROUPS[d])))]
    causal = bool(rng.integers(2))
    paged = bool(rng.integers(4))  # mostly paged
    B = int(rng.integers(1, 7))
    q_lens, kv_lens = [], []
    for _ in range(B):
        kind = rng.integers(3)
        if kind == 0:      # decode-like
            ql = int(rng.integers(1, 4))
        elif kind == 1:    # short prefill
            ql = int(rng.integers(4, 90))
        else:              # longer prefill
            ql = int(rng.integers(90, 420))
        L = ql + int(rng.integers(0, 2500))
        if not causal and rng.integers(4) == 0:
            L = int(rng.integers(1, max(2, ql)))  # fewer keys than queries
        q_lens.append(ql)
        kv_lens.append(max(L, 1))
    return d, hq, hkv, causal, paged, q_lens, kv_lens


@pytest.mark.parametrize("seed", list(range(48)))
def test_random_shapes(seed):
    d, hq, hkv, causal, paged, q_lens, kv_lens = _case(9000 + seed)
    if paged:
        wl = workloads.make_paged("fuzz", 9100 + seed, q_lens, kv_lens, hq, hkv, d, 64,
                                  causal=causal, extra_pages=3)
    else:
        wl = workloads.make_contiguous("fuzz", 9100 + seed, q_lens, kv_lens, hq, hkv, d, causal=causal)
    out = run_gpu(wl)
    assert_parity(out, wl)
    import paged_kv_flashattention_varlen_gb300 as pk
    assert pk.device_status() == 0


def _same_bits(a, b):
    return torch.equal(a.cpu().view(torch.int16), b.cpu().view(torch.int16))


@pytest.mark.parametrize("seed", list(range(16)))
def test_random_shapes_append(seed):
    """The cache write of the new tokens then attention (pattn_forward_append) on
    the same random shapes: the pool bit for bit against the oracle's write, the
    output over every row against the oracle."""
    import oracle
    import paged_kv_flashattention_varlen_gb300 as pk
    d, hq, hkv, causal, paged, q_lens, kv_lens = _case(9000 + seed)
    if paged:
        wl = workloads.make_paged("fuzz_app", 9200 + seed, q_lens, kv_lens, hq, hkv, d, 64, causal=causal,
                                  extra_pages=3)
    else:
        wl = workloads.make_contiguous("fuzz_app", 9200 + seed, q_lens, kv_lens, hq, hkv, d, causal=causal)
    k, v = workloads.new_kv_rows(wl, 9400 + seed)
    ref_wl = oracle.append_workload(wl, k, v)
    dev = to_device(wl)
    out = torch.full_like(dev["q"], float("nan"))
    pk.forward_append(out, dev["q"], k.to(dev["q"].device), v.to(dev["q"].device), dev["kv"], dev["bt"],
                      dev["sl"], dev["cu"], max_q=wl.max_q, max_kv=wl.max_kv, n_heads_kv=wl.n_heads_kv,
                      scale=wl.scale, causal=wl.causal, num_pages=wl.num_pages)
    torch.cuda.synchronize()
    assert pk.device_status() == 0
    assert _same_bits(dev["kv"], ref_wl.kv_pool), "cache after the write differs from the oracle's"
    assert_parity(out, ref_wl)
