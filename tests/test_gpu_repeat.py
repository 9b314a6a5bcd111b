"""Race detection by repetition: every path of the library is bitwise repeatable
for a fixed batch (the tile plan depends only on the lengths, KV splits are
merged in split order whichever CTA merges them, the K-mean sums are exact in
fixed point). A missing barrier, an mbarrier phase slip, a split counter read
before its partial rows land or a decode/prefill kernel overlap that touches
the other's workspace shows up as an output that differs in some run and not
in others. These tests issue many calls back to back on one stream, with no
host synchronisation between them (each call's kernels chained by dependent
launches, the next call's planner behind them), each into its own output
buffer, then compare every output with the first bit for bit and read the
device error word once at the end.

Shapes: the 64-sequence decode batch and the mixed decode + prefill-chunk
batch at full size (both kernels in one call, split units in each), the
2-sequence paged decode, a quarter of the 4 x 8192 causal prefill, and the
quantised and cache-write entry points on smaller cuts of the same shapes.
"""
import pytest
import torch

import workloads
from helpers import to_device

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

REPEATS = 24


def _bits(t):
    return t.view(torch.int16)


def _issue(fn, wl, d, n):
    outs = [torch.full_like(d["q"], float("nan")) for _ in range(n)]
    for out in outs:
        fn(out, wl, d)
    torch.cuda.synchronize()
    return outs


def _forward(out, wl, d):
    import paged_kv_flashattention_varlen_gb300 as pk
    pk.forward(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q, max_kv=wl.max_kv,
               n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal, num_pages=wl.num_pages)


def _fp8qk(out, wl, d):
    import paged_kv_flashattention_varlen_gb300 as pk
    pk.forward_fp8qk(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q,
                     max_kv=wl.max_kv, n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                     num_pages=wl.num_pages)


def _fp8(out, wl, d):
    import paged_kv_flashattention_varlen_gb300 as pk
    pk.forward_fp8(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q,
                   max_kv=wl.max_kv, n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                   num_pages=wl.num_pages)


def _append(out, wl, d):
    # the same new rows every call: after the first call each write stores the
    # values already in the pool, so every attention reads the same cache
    import paged_kv_flashattention_varlen_gb300 as pk
    pk.forward_append(out, d["q"], d["k_new"], d["v_new"], d["kv"], d["bt"], d["sl"], d["cu"],
                      max_q=wl.max_q, max_kv=wl.max_kv, n_heads_kv=wl.n_heads_kv, scale=wl.scale,
                      causal=wl.causal, num_pages=wl.num_pages)


CASES = {
    "decode_batch": (lambda: workloads.named(2), _forward),
    "mixed_d256": (lambda: workloads.named(5), _forward),
    "tiny_decode_d256": (lambda: workloads.named(1), _forward),
    "causal_prefill": (lambda: workloads.named(3, scale_down=4), _forward),
    "noncausal_contiguous": (lambda: workloads.named(4, scale_down=8), _forward),
    "fp8qk_prefill": (lambda: workloads.named(3, scale_down=8), _fp8qk),
    "fp8_prefill": (lambda: workloads.named(3, scale_down=8), _fp8),
    "append_decode_batch": (lambda: workloads.named(2, scale_down=4), _append),
    "append_mixed_d256": (lambda: workloads.named(5, scale_down=4), _append),
}


@pytest.mark.parametrize("name", list(CASES))
def test_back_to_back_calls_are_bitwise_equal(name):
    import paged_kv_flashattention_varlen_gb300 as pk
    make, fn = CASES[name]
    wl = make()
    d = to_device(wl)
    if fn is _append:
        k, v = workloads.new_kv_rows(wl, seed=11)
        d["k_new"], d["v_new"] = k.cuda(), v.cuda()
    assert pk.device_status() == 0
    outs = _issue(fn, wl, d, REPEATS)
    assert pk.device_status() == 0
    ref = _bits(outs[0])
    assert torch.isfinite(outs[0].float()).all()
    differing = [i for i, o in enumerate(outs[1:], 1) if not torch.equal(_bits(o), ref)]
    assert not differing, f"calls {differing} differ from the first"
