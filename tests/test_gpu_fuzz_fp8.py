"""GPU parity of the two quantised modes on seeded random shapes (head_dim 128):
the e4m3 Q/K codes and scales (and V codes and scales for the fp8 P.V mode)
bit for bit against oracle/quant.py, and the output rows of prefill units
against the oracle of each mode (the attention over dequantised Q and K within
the parity bar; the fp8 P.V method within its probability-rounding bound).
Units of at most 16 packed query rows run on the bf16 decode kernel in both
modes and are compared with the float64 oracle of the plain method."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import MAX_ABS, MEAN_ABS, to_device
from oracle import quant

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_flashattention_varlen_gb300 import build
    build.build()


def _case(seed):
    rng = np.random.default_rng(seed)
    hq, hkv = [(4, 1), (8, 2), (16, 4), (32, 4), (8, 8)][int(rng.integers(5))]
    causal = bool(rng.integers(2))
    paged = bool(rng.integers(4))
    q_lens, kv_lens = [], []
    for _ in range(int(rng.integers(1, 5))):
        ql = int(rng.integers(1, 3)) if rng.integers(3) == 0 else int(rng.integers(4, 260))
        q_lens.append(ql)
        kv_lens.append(ql + int(rng.integers(0, 1500)))
    if paged:
        return workloads.make_paged("fuzz8", 9300 + seed, q_lens, kv_lens, hq, hkv, 128, 64, causal=causal,
                                    extra_pages=2)
    return workloads.make_contiguous("fuzz8", 9300 + seed, q_lens, kv_lens, hq, hkv, 128, causal=causal)


def _rows(wl):
    """(decode-unit rows, prefill-unit rows): a unit of at most 16 packed rows
    runs on the decode kernel."""
    G = wl.n_heads_q // wl.n_heads_kv
    cu = wl.cu_q.numpy()
    dec, pre = [], []
    for b in range(wl.num_seqs):
        ql = int(cu[b + 1] - cu[b])
        (dec if ql * G <= 16 else pre).extend(range(int(cu[b]), int(cu[b + 1])))
    return dec, pre


def _check_bar(got, ref):
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())


@pytest.mark.parametrize("seed", list(range(12)))
def test_random_shapes_fp8qk(seed):
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = _case(seed)
    d = to_device(wl)
    q8, qs, k8, ks = pk.quantize_qk(d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q,
                                     max_kv=wl.max_kv, n_heads_kv=wl.n_heads_kv, num_pages=wl.num_pages)
    torch.cuda.synchronize()
    ref = quant.quantize_workload(wl)
    assert np.array_equal(q8.cpu().numpy(), ref["q_codes"])
    assert np.array_equal(qs.cpu().numpy().view(np.uint32), ref["q_scale"].view(np.uint32))
    nb = k8.shape[0] // wl.num_seqs
    k8c, ksc = k8.cpu().numpy(), ks.cpu().numpy()
    for b in range(wl.num_seqs):
        kc, kss = ref["k_codes"][b], ref["k_scale"][b]
        nblk = kss.shape[0]
        assert np.array_equal(k8c[b * nb:b * nb + nblk].reshape(nblk * 64, wl.n_heads_kv, 128), kc)
        assert np.array_equal(ksc[b * nb:b * nb + nblk].view(np.uint32), kss.view(np.uint32))
    out = torch.full_like(d["q"], float("nan"))
    pk.forward_fp8qk(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q, max_kv=wl.max_kv,
                     n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal, num_pages=wl.num_pages)
    torch.cuda.synchronize()
    assert pk.device_status() == 0
    dec, pre = _rows(wl)
    if pre:
        got = out[torch.as_tensor(pre, device=out.device)].float().cpu().numpy()
        _check_bar(got, quant.attention_dequantized(wl, rows=pre))
    if dec:
        got = out[torch.as_tensor(dec, device=out.device)].float().cpu().numpy()
        _check_bar(got, oracle.forward_workload(wl, rows=dec)[0])


@pytest.mark.parametrize("seed", list(range(12)))
def test_random_shapes_fp8(seed):
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = _case(seed)
    d = to_device(wl)
    out = torch.full_like(d["q"], float("nan"))
    pk.forward_fp8(out, d["q"], d["kv"], d["bt"], d["sl"], d["cu"], max_q=wl.max_q, max_kv=wl.max_kv,
                   n_heads_kv=wl.n_heads_kv, scale=wl.scale, causal=wl.causal, num_pages=wl.num_pages)
    torch.cuda.synchronize()
    assert pk.device_status() == 0
    dec, pre = _rows(wl)
    if pre:
        got = out[torch.as_tensor(pre, device=out.device)].float().cpu().numpy()
        ref, bound = quant.attention_fp8(wl, rows=pre)
        assert np.isfinite(got).all()
        err = np.abs(got - ref)
        assert (err / bound).max() <= 1.0, ((err / bound).max(), err.max())
        assert err.mean() <= 0.1 * bound.mean(), (err.mean(), bound.mean())
    if dec:
        got = out[torch.as_tensor(dec, device=out.device)].float().cpu().numpy()
        _check_bar(got, oracle.forward_workload(wl, rows=dec)[0])
