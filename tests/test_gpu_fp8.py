"""GPU parity of the fp8 P.V variant (pattn_quantize_v, pattn_forward_fp8)
against oracle/quant.py: the transposed e4m3 V codes and per-channel scales bit
for bit, and the output within the per-element bound of e4m3 probabilities
around the float64 attention over the dequantised Q, K and V (tight where
every probability is exact)."""
import numpy as np
import pytest
import torch

import workloads
from helpers import sample_rows, to_device
from oracle import quant

pytestmark = pytest.mark.gpu


def _cases():
    return {
        "paged_causal": workloads.named(3, scale_down=16),                        # 4 x 512, G 4
        "contig_noncausal_offset": workloads.named(4, scale_down=32),             # K channel offsets
        "paged_varlen": workloads.make_paged("varlen8", 61, [17, 200, 64, 1], [300, 200, 1000, 129],
                                             16, 4, 128, causal=True, extra_pages=5),
    }


def _run(wl, d):
    import paged_kv_flashattention_varlen_gb300 as pk
    out = torch.full_like(d["q"], float("nan"))
    pk.forward_fp8(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q, max_kv=wl.max_kv,
                   n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal, num_pages=wl.num_pages)
    torch.cuda.synchronize()
    assert pk.device_status() == 0
    return out


def _within_bound(got, ref, bound):
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    worst = (err / bound).max()
    assert worst <= 1.0, (worst, err.max(), err.mean())
    return err


@pytest.mark.parametrize("name", ["paged_causal", "contig_noncausal_offset", "paged_varlen"])
def test_v_codes_and_scales_bitwise(name):
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = _cases()[name]
    d = to_device(wl)
    v8, vs = pk.quantize_v(d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q, max_kv=wl.max_kv,
                           n_heads_kv=wl.n_heads_kv, num_pages=wl.num_pages)
    torch.cuda.synchronize()
    assert pk.device_status() == 0
    nt = v8.shape[0] // wl.num_seqs
    v8c, vsc = v8.cpu().numpy(), vs.cpu().numpy()
    start = 0
    for b in range(wl.num_seqs):
        v32 = quant.logical_v(wl.kv_pool, wl.block_table, wl.seq_lens, b, wl.page_size, start)
        start += int(wl.seq_lens[b])
        codes, scale = quant.quantize_v(v32)
        assert np.array_equal(v8c[b * nt:b * nt + codes.shape[0]], codes), f"sequence {b}: V codes"
        assert np.array_equal(vsc[b].view(np.uint32), scale.view(np.uint32)), f"sequence {b}: V scales"


@pytest.mark.parametrize("name", ["paged_causal", "contig_noncausal_offset", "paged_varlen"])
def test_attention_within_the_probability_rounding_bound(name):
    wl = _cases()[name]
    out = _run(wl, to_device(wl))
    rows = sample_rows(wl, per_seq=8)
    ref, bound = quant.attention_fp8(wl, rows=rows)
    got = out[torch.as_tensor(rows, device=out.device)].float().cpu().numpy()
    err = _within_bound(got, ref, bound)
    # the rounding errors of P are unbiased: far below the worst case on average
    assert err.mean() <= 0.1 * bound.mean(), (err.mean(), bound.mean())


@pytest.mark.parametrize("causal", [True, False])
def test_group_of_eight_ragged_lengths(causal):
    # G 8 (16 tokens per q tile), lengths around the 64-key blocks and 128-key tiles
    wl = workloads.make_paged("fp8g8", 63 + causal, [1, 65, 129, 200, 16], [1, 65, 1000, 200, 3000], 32, 4, 128,
                              causal=causal, extra_pages=3)
    out = _run(wl, to_device(wl))
    rows = sample_rows(wl, per_seq=10)
    ref, bound = quant.attention_fp8(wl, rows=rows)
    got = out[torch.as_tensor(rows, device=out.device)].float().cpu().numpy()
    _within_bound(got, ref, bound)


def test_equal_keys_give_the_exact_mean_of_the_values():
    # every key of a head equal: smoothed K is zero, every score 0 and every
    # p * 2^2 = 4 exact in e4m3, so the output is the mean of the dequantised V
    # rows up to fp32 sums and the bf16 output
    wl = workloads.make_paged("eqk", 62, [40, 300, 7], [300, 700, 129], 16, 4, 128, causal=True,
                              extra_pages=3)
    rng = np.random.default_rng(5)
    krow = torch.from_numpy(rng.standard_normal((4, 128)).astype(np.float32)).to(torch.bfloat16)
    wl.kv_pool[:, 0] = krow[None, None]
    out = _run(wl, to_device(wl))
    rows = sample_rows(wl, per_seq=12)
    ref, _ = quant.attention_fp8(wl, rows=rows)
    got = out[torch.as_tensor(rows, device=out.device)].float().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


def test_full_size_noncausal_sampled_rows():
    """The 37,810-token non-causal shape (one sequence, 56 heads) on sampled rows."""
    wl = workloads.named(4)
    out = _run(wl, to_device(wl))
    rows = [0, 1, 127, 128, 18905, 37808, 37809]
    ref, bound = quant.attention_fp8(wl, rows=rows)
    got = out[torch.as_tensor(rows, device=out.device)].float().cpu().numpy()
    _within_bound(got, ref, bound)


def test_decode_units_take_the_bf16_decode_kernel():
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = workloads.named(2, scale_down=8)
    d = to_device(wl)
    a = _run(wl, d)
    b = torch.full_like(d["q"], float("nan"))
    pk.forward(b, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q, max_kv=wl.max_kv,
               n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal, num_pages=wl.num_pages)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_unsupported_head_dim():
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = workloads.named(1)  # head_dim 256
    d = to_device(wl)
    out = torch.empty_like(d["q"])
    rc = pk.forward_fp8(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q,
                        max_kv=wl.max_kv, n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal,
                        num_pages=wl.num_pages, check=False)
    assert rc == 2
