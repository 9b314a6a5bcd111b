"""Pins for the quantised-QK oracle (CPU only): the e4m3 format from its
definition, the scale rule, the block layout of the K codes, the smoothing
invariance, and the dequantised attention against the C oracle where the
quantisation is exact."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import quant


def e4m3_from_definition(code: int) -> float:
    """Value of an e4m3 byte: sign, 4 exponent bits (bias 7), 3 mantissa bits;
    exponent 0 is subnormal; 0x7F / 0xFF are NaN."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_e4m3_values_match_the_format_definition():
    codes = np.arange(256, dtype=np.uint8)
    got = quant.e4m3_values(codes)
    for c in range(256):
        want = e4m3_from_definition(c)
        if math.isnan(want):
            assert math.isnan(got[c])
        else:
            assert got[c] == want, c


@pytest.mark.parametrize("x,code", [
    (0.0, 0x00), (1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (1000.0, 0x7E), (-1000.0, 0xFE),
    (2.0 ** -9, 0x01),                      # smallest subnormal
    (1.0625, 0x38), (1.1875, 0x3A),          # ties go to the even mantissa
    (1.0625 + 1e-6, 0x39), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02),
])
def test_e4m3_rounding(x, code):
    assert int(quant.e4m3_codes(np.array([x], dtype=np.float32))[0]) == code


def test_codes_are_nearest_and_saturated():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(4096) * 100).astype(np.float32)
    c = quant.e4m3_codes(x)
    v = quant.e4m3_values(c)
    grid = np.array(sorted({e4m3_from_definition(k) for k in range(256) if not math.isnan(e4m3_from_definition(k))}))
    clipped = np.clip(x.astype(np.float64), -448, 448)
    nearest = grid[np.abs(grid[None, :] - clipped[:, None]).argmin(axis=1)]
    assert np.all(np.abs(v - clipped) <= np.abs(nearest - clipped) + 0.0)


def test_row_scale_maps_amax_to_448_and_zero_rows_to_zero():
    q = np.zeros((3, 2, 128), dtype=np.float32)
    q[0, 0, 5] = -3.25
    q[0, 0, 7] = 1.0
    q[1, 1] = np.linspace(-2, 7, 128, dtype=np.float32)
    codes, s = quant.quantize_q(q)
    assert s[0, 0] == np.float32(3.25) / np.float32(448)
    assert quant.e4m3_values(codes[0, 0, 5:6])[0] == -448.0
    assert s[2, 0] == 1.0 and not codes[2].any()
    assert quant.e4m3_values(codes[1, 1]).max() == 448.0


def test_codes_dequantise_within_half_an_e4m3_step():
    # code * scale is x up to the e4m3 rounding (relative 2^-4 for normal codes,
    # absolute 2^-10 * scale for subnormal ones) plus fp32 slack from the
    # multiplier, and the row maximum maps to +-448
    rng = np.random.default_rng(8)
    q = (rng.standard_normal((64, 4, 128)) * rng.uniform(0.01, 50, (64, 4, 1))).astype(np.float32)
    codes, s = quant.quantize_q(q)
    deq = quant.e4m3_values(codes) * s[:, :, None].astype(np.float64)
    bound = np.maximum(np.abs(q) * 2.0 ** -4, 2.0 ** -10 * s[:, :, None]) * (1 + 1e-5)
    assert np.all(np.abs(deq - q) <= bound)
    vmax = np.abs(quant.e4m3_values(codes)).max(axis=2)
    assert np.all(vmax == 448.0)


def test_tiny_and_nan_rows_give_finite_codes():
    q = np.zeros((3, 1, 128), dtype=np.float32)
    q[0, 0, :4] = [1e-39, -5e-40, 0.0, 2e-45]   # 448 / amax overflows fp32: capped
    q[1, 0, :3] = [np.nan, 2.0, -1.0]           # NaN ignored by amax
    codes, s = quant.quantize_q(q)
    vals = quant.e4m3_values(codes)
    assert np.isfinite(vals[0]).all() and s[0, 0] == np.float32(1e-39) / np.float32(448)
    assert s[1, 0] == np.float32(2.0) / np.float32(448) and vals[1, 0, 1] == 448.0
    assert np.isnan(vals[1, 0, 0])               # the NaN element itself stays NaN
    assert not codes[2].any() and s[2, 0] == 1.0


def test_k_blocks_of_64_keys_and_zero_tail():
    rng = np.random.default_rng(5)
    k = rng.standard_normal((100, 2, 128)).astype(np.float32)
    m = quant.k_mean(k)
    assert m.dtype == np.float32
    assert np.allclose(m, k.astype(np.float64).mean(axis=0), atol=1e-7)
    codes, scales = quant.quantize_k(k, m)
    assert codes.shape == (128, 2, 128) and scales.shape == (2, 2)
    assert not codes[100:].any()
    x = k - m[None]
    assert scales[1, 0] == np.float32(np.abs(x[64:100, 0]).max()) / np.float32(448)


def test_k_mean_is_the_plain_mean_for_keys_on_the_grid():
    # bf16 keys of magnitude 2^-25 ... 1024 lie on the 2^-32 grid, so the
    # fixed-point sum is the exact sum and the offset is the fp32-rounded mean
    rng = np.random.default_rng(11)
    k = torch.from_numpy(rng.standard_normal((333, 3, 128)) * 50).to(torch.bfloat16).float().numpy()
    k = np.where(np.abs(k) < 2.0 ** -25, 0.0, k).astype(np.float32)
    k[0, 0, 0] = 1024.0
    k[1, 0, 0] = -1024.0
    exact = np.array([[sum(float(v) for v in k[:, h, c]) for c in range(128)] for h in range(3)])
    assert np.array_equal(quant.k_sum_units(k), (exact * 2.0 ** 32).astype(np.int64))
    assert np.array_equal(quant.k_mean(k), (exact / 333).astype(np.float32))


def test_k_sum_clamps_and_rounds_to_the_grid():
    k = np.zeros((6, 1, 128), dtype=np.float32)
    k[0, 0, 0] = 4096.0                 # clamped to 1024
    k[1, 0, 0] = -3.0e38                # clamped to -1024
    k[2, 0, 1] = 2.0 ** -33             # half a unit: ties to even -> 0
    k[3, 0, 1] = 3 * 2.0 ** -33         # one and a half units -> 2
    k[4, 0, 2] = 2.0 ** -30             # 4 units, exact
    k[5, 0, 2] = -(2.0 ** -34)          # a quarter unit -> 0
    k[0, 0, 3] = np.nan                 # NaN counts as the lower bound
    units = quant.k_sum_units(k)[0]
    assert units[0] == 0 and units[1] == 2 and units[2] == 4
    assert units[3] == -1024 * 2 ** 32
    assert quant.k_mean(k)[0, 2] == np.float32(4 * 2.0 ** -32 / 6)


def test_exact_quantisation_reproduces_the_plain_attention():
    # values on the e4m3 grid with a power-of-two row maximum of 448 * 2^-6, and
    # K in +- pairs per channel (zero mean): the codes are exact, so the
    # dequantised attention must equal the float64 C oracle on the same inputs
    rng = np.random.default_rng(7)
    grid = np.array([0.0, 0.25, 0.5, 1.0, 1.5, 2.0, 3.0, 448.0])
    T, Hq, Hkv, D, L = 4, 4, 2, 128, 64
    q = rng.choice(grid, size=(T, Hq, D)) * rng.choice([-1, 1], size=(T, Hq, D))
    q[..., 0] = 448.0
    half = rng.choice(grid[:-1], size=(L // 2, Hkv, D)) * rng.choice([-1, 1], size=(L // 2, Hkv, D))
    k = np.concatenate([half, -half], axis=0)
    k[0, :, 1] = 448.0
    k[L // 2, :, 1] = -448.0
    scale_pow = 2.0 ** -6
    q *= scale_pow
    k *= scale_pow
    wl = workloads.make_paged("exactq", 3, [T], [L], Hq, Hkv, D, causal=True, extra_pages=1)
    wl.q.copy_(torch.from_numpy(q).to(torch.bfloat16))
    page = int(wl.block_table[0, 0])
    wl.kv_pool[page, 0, :L].copy_(torch.from_numpy(k).to(torch.bfloat16))
    qz = quant.quantize_workload(wl)
    assert np.array_equal(quant.e4m3_values(qz["q_codes"]) * qz["q_scale"][:, :, None], q)
    assert np.array_equal(qz["k_mean"][0], np.zeros((Hkv, D), np.float32))
    got = quant.attention_dequantized(wl, qz=qz)
    ref, _ = oracle.forward_workload(wl)
    assert np.abs(got - ref).max() < 1e-12


def test_smoothing_keeps_channel_offsets_out_of_the_error():
    # K with a large per-channel offset: with the mean removed the quantised
    # attention stays close to the exact one
    wl = workloads.make_contiguous("smooth", 9, [40], [300], 8, 2, 128, causal=False, k_offset_std=4.0)
    ref, _ = oracle.forward_workload(wl)
    got = quant.attention_dequantized(wl)
    err = np.abs(got - ref)
    assert err.max() < 0.1 and err.mean() < 0.01, (err.max(), err.mean())


# ---------------------------------------------------------------------------
# fp8 P.V: V codes and the error bound of the e4m3 probabilities


def test_v_codes_layout_scale_and_padding():
    rng = np.random.default_rng(21)
    L, H, D = 130, 2, 128
    v = torch.from_numpy(rng.standard_normal((L, H, D)) * 3).to(torch.bfloat16).float().numpy()
    v[:, 1, 7] = 0.0                                   # an all-zero channel
    codes, scale = quant.quantize_v(v)
    assert codes.shape == (2, H, D, 128) and scale.shape == (H, D)
    assert scale[1, 7] == 1.0 and not codes[:, 1, 7].any()
    amax = np.abs(v[:, 0, 3]).max()
    assert scale[0, 3] == np.float32(amax) / np.float32(448)
    # key j of tile t sits at codes[t, hk, d, j]; rows past L are zero codes
    for (j, hk, d) in [(0, 0, 0), (129, 1, 127), (64, 0, 5), (127, 1, 64)]:
        inv = np.float32(448) / np.float32(np.abs(v[:, hk, d]).max())
        want = quant.e4m3_codes(np.array([np.float32(v[j, hk, d]) * inv], dtype=np.float32))[0]
        assert codes[j // 128, hk, d, j % 128] == want
    assert not codes[1, :, :, 2:].any()
    # the channel maximum maps to +-448
    assert np.all(np.abs(quant.e4m3_values(codes)).max(axis=(0, 3))[0] == 448.0)


def test_v_on_the_e4m3_grid_dequantises_exactly():
    rng = np.random.default_rng(22)
    grid = np.array([0.0, 0.5, 1.0, 1.75, 3.0, 6.5, 448.0])
    v = rng.choice(grid, size=(70, 1, 128)) * rng.choice([-1, 1], size=(70, 1, 128))
    v[3, 0, :] = 448.0
    v *= 2.0 ** -5
    codes, scale = quant.quantize_v(v.astype(np.float32))
    assert np.array_equal(quant.dequantize_v(codes, scale, 70), v)


def test_exactly_coded_inputs_give_the_plain_attention():
    # Q, K and V on the e4m3 grid with power-of-two block maxima and zero-mean K:
    # every code is exact, so the oracle's fp8 output is the float64 C oracle's
    rng = np.random.default_rng(23)
    grid = np.array([0.0, 0.25, 0.5, 1.0, 1.5, 2.0, 3.0, 448.0])
    T, Hq, Hkv, D, L = 4, 4, 2, 128, 64
    q = rng.choice(grid, size=(T, Hq, D)) * rng.choice([-1, 1], size=(T, Hq, D))
    q[..., 0] = 448.0
    half = rng.choice(grid[:-1], size=(L // 2, Hkv, D)) * rng.choice([-1, 1], size=(L // 2, Hkv, D))
    k = np.concatenate([half, -half], axis=0)
    k[0, :, 1] = 448.0
    k[L // 2, :, 1] = -448.0
    v = rng.choice(grid[:-1], size=(L, Hkv, D)) * rng.choice([-1, 1], size=(L, Hkv, D))
    v[5] = 448.0
    q, k, v = q * 2.0 ** -6, k * 2.0 ** -6, v * 2.0 ** -7
    wl = workloads.make_paged("exactv", 3, [T], [L], Hq, Hkv, D, causal=True, extra_pages=1)
    wl.q.copy_(torch.from_numpy(q).to(torch.bfloat16))
    page = int(wl.block_table[0, 0])
    wl.kv_pool[page, 0, :L].copy_(torch.from_numpy(k).to(torch.bfloat16))
    wl.kv_pool[page, 1, :L].copy_(torch.from_numpy(v).to(torch.bfloat16))
    got, bound = quant.attention_fp8(wl)
    ref, _ = oracle.forward_workload(wl)
    assert np.abs(got - ref).max() < 1e-12
    assert np.all(bound > 0)


def test_bound_covers_simulated_probability_rounding():
    # round every p * 2^(2 + d) to e4m3 for a trailing max d in [0, 6] (fp32
    # row sum of the unrounded p): the output error stays within the bound
    rng = np.random.default_rng(24)
    for n in [1, 2, 3, 7, 64, 300, 5000]:
        for trial in range(20):
            s = rng.standard_normal(n) * rng.uniform(0.5, 6)
            v = rng.standard_normal((n, 16)) * rng.uniform(0.1, 4)
            w = np.exp(s - s.max())
            d = rng.uniform(0, quant.P_SLACK_LOG2)
            scaled = w * 2.0 ** (P := quant.P_SCALE_LOG2) * 2.0 ** d
            ph = quant.e4m3_values(quant.e4m3_codes(scaled.astype(np.float32)))
            o_hat = (ph @ v) / scaled.sum()
            o = (w @ v) / w.sum()
            bnd = ((2.0 ** -4) * (w @ np.abs(v)) + (2.0 ** -(10 + P)) * np.abs(v).sum(0)) / w.sum()
            assert np.all(np.abs(o_hat - o) <= bnd * (1 + 1e-6) + 1e-12), (n, trial)
    assert P == 2 and quant.P_SLACK_LOG2 + quant.P_SCALE_LOG2 <= 8   # codes <= 2^8 < 448
