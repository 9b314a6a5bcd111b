"""pattn_forward inside a CUDA graph.

Once the library workspace exists (a first call outside the capture), a call
records only kernel launches on the caller's stream: the plan is made on the
device from the device data at every replay, so a captured call follows
new lengths, offsets and block tables written into the same buffers between
replays (within the bounds given at capture). Each replay is compared bit for
bit with an eager call on the same data, and with the float64 oracle.
"""
import numpy as np
import pytest
import torch

import workloads
from helpers import assert_parity, to_device

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_flashattention_varlen_gb300 import build
    build.build()


def _call(pk, wl, d, out):
    pk.forward(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q, max_kv=wl.max_kv,
               n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal, num_pages=wl.num_pages)


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("which", ["decode_batch", "causal_prefill", "mixed_d256"])
def test_replays_match_eager_calls_bitwise(which):
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = {"decode_batch": lambda: workloads.named(2, scale_down=4),
          "causal_prefill": lambda: workloads.named(3, scale_down=16),
          "mixed_d256": lambda: workloads.named(5, scale_down=8)}[which]()
    d = to_device(wl)
    ref = torch.full_like(d["q"], float("nan"))
    _call(pk, wl, d, ref)  # eager, and the workspace now exists
    torch.cuda.synchronize()
    out = torch.full_like(d["q"], float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _call(pk, wl, d, out)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert _same_bits(out, ref)
    assert pk.device_status() == 0


def test_a_captured_call_follows_new_lengths_written_between_replays():
    # one capture of a decode batch; between replays the sequences' KV lengths
    # are rewritten in place (within max_kv): the device plan of each replay
    # follows them, and each replay equals an eager call on the new lengths
    import paged_kv_flashattention_varlen_gb300 as pk
    rng = np.random.default_rng(4)
    lens = rng.integers(300, 5000, size=24)
    wl = workloads.make_paged("graph_lens", 91, [1] * 24, lens.tolist(), 32, 8, 128, 64, causal=True,
                              extra_pages=4)
    d = to_device(wl)
    out = torch.full_like(d["q"], float("nan"))
    _call(pk, wl, d, out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _call(pk, wl, d, out)
    for step in range(3):
        # shorter sequences: each keeps a prefix of its pages (the tail rows of
        # its new last page hold real keys now, masked by the new length)
        new_lens = np.maximum(1, lens - rng.integers(0, 1200, size=lens.size)).astype(np.int32)
        d["sl"].copy_(torch.from_numpy(new_lens))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref = torch.full_like(out, float("nan"))
        _call(pk, wl, d, ref)
        torch.cuda.synchronize()
        assert _same_bits(out, ref), step
        new_wl = workloads.Workload(**{**wl.__dict__, "seq_lens": torch.from_numpy(new_lens)})
        assert_parity(out, new_wl)
    assert pk.device_status() == 0
