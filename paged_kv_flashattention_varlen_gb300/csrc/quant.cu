// quant.cu -- the preparation phases of the quantised-QK variant (the GB10
// "sage2" benchmark page: k_mean_and_smoothing_preparation,
// q_int8_quantization, k_int8_subtract_mean_quantization), with fp8 e4m3 codes
// in place of int8: on sm_103a the e4m3 tensor-core rate is twice the bf16 one
// and the int8 rate is far below it.
//
//   * k_sum_kernel: per (sequence, KV head, channel), the sum of the sequence's
//     keys in fixed point: each key value clamped to +-1024 and rounded to the
//     2^-32 grid (exact for |x| >= 2^-25), as an int64 count. Each CTA adds up
//     256 keys in int32 lanes and adds its partial sums with 64-bit integer
//     atomics; the sums are exact, so the order does not matter. The CTA that
//     finishes last for its (sequence, KV head) turns the sums into the fp32
//     smoothing offsets (sum * 2^-32 / L in float64, rounded to fp32).
//   * k_quant_kernel: per (sequence, 64-key block, KV head): x = k - offset in
//     fp32, amax = max |x|, scale = amax / 448, inv = 448 / amax (IEEE
//     divisions, once per block; inv capped at the largest finite fp32; 1 and 1
//     when amax = 0), code = e4m3 round-to-nearest-even of x * inv, saturated.
//     Rows past L are zero codes.
//   * q_quant_kernel: per query row (token, head): scale and codes as above.
//   * V (fp8 P.V variant): k_sum_kernel also takes max |v| per (sequence, KV
//     head, channel), and its last CTA writes scale = amax / 448 and
//     inv = 448 / amax; v_quant_kernel writes code = e4m3(v * inv) per 128-key
//     tile and head, transposed through shared memory to [channel][key] (the
//     K-major B operand of the P.V MMA), with zero codes past the sequence end.
//
// Every rounding decision is taken in the precision the oracle uses, so codes
// and scales agree with it bit for bit. The kernels run after the plan (they
// read its validated lengths and contiguous row offsets and skip rejected
// sequences) and before the attention kernel, as dependent launches.
#include <cuda_fp8.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace pattn {
namespace {

constexpr int kSumKeys = 256;  // keys per k_sum CTA
constexpr float kE4m3Max = 448.0f;
constexpr float kSumClamp = 1024.0f;            // key values are clamped to +-1024 for the sum
constexpr float kSumUnit = 4294967296.0f;       // 2^32: the sum counts units of 2^-32
constexpr float kSplitBias = 26388279066624.0f; // 1.5 * 2^44: x + it rounds x to a multiple of 2^21
constexpr float kIntBias = 12582912.0f;         // 1.5 * 2^23: x + it rounds x to an integer
constexpr int kIntBiasBits = 0x4B400000;        // the fp32 bits of 1.5 * 2^23
constexpr float kHiStep = 4.76837158203125e-07f;  // 2^-21

// Adds two key values (a bf16 pair) to per-channel int32 counters, exactly.
// With u = clamp(v, +-1024) * 2^32 (exact, |u| <= 2^42): u_hi = u rounded to a
// multiple of 2^21 and u_lo = u - u_hi (exact, |u_lo| <= 2^20), so that
// round(u) = u_hi + round(u_lo), ties to even (u_hi is even). u_hi / 2^21 and
// round(u_lo) are read off the bits of t + 1.5 * 2^23, whose fp32 grid there
// is the integers; the bias is taken off in the same integer add.
__device__ __forceinline__ void add_units(uint32_t pair, int& hi0, int& lo0, int& hi1, int& lo1) {
  __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&pair);
  v = __hmin2(__hmax2(v, __float2bfloat162_rn(-kSumClamp)), __float2bfloat162_rn(kSumClamp));
  const float2 f = __bfloat1622float2(v);
  const float2 unit = make_float2(kSumUnit, kSumUnit);
  const float2 t = __ffma2_rn(f, unit, make_float2(kSplitBias, kSplitBias));
  const float2 uh = __fadd2_rn(t, make_float2(-kSplitBias, -kSplitBias));
  const float2 ul = __ffma2_rn(f, unit, make_float2(-uh.x, -uh.y));
  const float2 a = __fadd2_rn(ul, make_float2(kIntBias, kIntBias));
  const float2 h = __ffma2_rn(uh, make_float2(kHiStep, kHiStep), make_float2(kIntBias, kIntBias));
  lo0 += __float_as_int(a.x) - kIntBiasBits;
  lo1 += __float_as_int(a.y) - kIntBiasBits;
  hi0 += __float_as_int(h.x) - kIntBiasBits;
  hi1 += __float_as_int(h.y) - kIntBiasBits;
}

__device__ __forceinline__ float e4m3_scale(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
}

// The quantisation multiplier 448 / amax (capped at the largest finite fp32; 1 for amax = 0).
__device__ __forceinline__ float e4m3_inv_scale(float amax) {
  return amax > 0.f ? fminf(__fdiv_rn(kE4m3Max, amax), 3.402823466e38f) : 1.0f;
}

// Two fp32 values -> two e4m3 bytes (first value in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Pointer to the K (plane 0) or V (plane 1) row j of sequence b, KV head hk
// (nullptr if its page is not a pool page; the plan has then rejected the
// sequence already). A contiguous cache holds num_pages rows per plane.
__device__ __forceinline__ const __nv_bfloat16* kv_row(const QuantParams& p, int b, int4 si, int j, int hk,
                                                       int plane) {
  const size_t row = static_cast<size_t>(p.n_heads_kv) * p.head_dim;
  if (p.block_table) {
    const int page = p.block_table[static_cast<size_t>(b) * p.bt_stride + j / kPage];
    if (page < 0 || page >= p.num_pages) return nullptr;
    return p.kv_pool + ((static_cast<size_t>(page) * 2 + plane) * kPage + (j % kPage)) * row +
           static_cast<size_t>(hk) * p.head_dim;
  }
  return p.kv_pool + (static_cast<size_t>(plane) * p.num_pages + si.w + j) * row +
         static_cast<size_t>(hk) * p.head_dim;
}
__device__ __forceinline__ const __nv_bfloat16* key_row(const QuantParams& p, int b, int4 si, int j, int hk) {
  return kv_row(p, b, si, j, hk, 0);
}

// grid (num_seqs * n_heads_kv, key chunks of kSumKeys), 256 threads: thread t
// adds channels 8 (t % 16) ... + 7 of keys j0 + t / 16, + 16, ... (16-byte
// loads, four keys of a lane in flight) and, when V codes are wanted, takes
// the max |v| of the same rows; the 16 key lanes are then combined in shared
// memory and the CTA adds its 128 partial sums with int64 atomics (and its
// maxima with uint32 atomic max on the fp32 bits, which order like the values
// for non-negative floats). The last CTA of a (sequence, KV head) writes the
// 128 K offsets and V scales.
__global__ void __launch_bounds__(256) k_sum_kernel(const QuantParams p) {
  grid_dep_launch();
  grid_dep_wait();  // the plan is complete
  __shared__ long long s_part[16][128];
  __shared__ float s_vmax[16][128];
  __shared__ int s_last;
  const int b = blockIdx.x / p.n_heads_kv, hk = blockIdx.x % p.n_heads_kv;
  const int4 si = p.seq_info[b];
  if (si.y < 0) return;
  const int L = si.z;
  const int j0 = blockIdx.y * kSumKeys, j1 = min(L, j0 + kSumKeys);
  if (j0 >= j1) return;
  const bool want_v = p.v8 != nullptr;
  const int cg = threadIdx.x & 15, kl = threadIdx.x >> 4;
  int hi[8], lo[8];
  float vmax[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    hi[e] = lo[e] = 0;
    vmax[e] = 0.f;
  }
  for (int jb = j0; jb < j1; jb += 64) {
    uint4 raw[4], rv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = jb + u * 16 + kl;
      const __nv_bfloat16* r = j < j1 ? key_row(p, b, si, j, hk) : nullptr;
      raw[u] = r ? *reinterpret_cast<const uint4*>(r + cg * 8) : make_uint4(0, 0, 0, 0);
      if (want_v) {
        const __nv_bfloat16* rv_ptr = j < j1 ? kv_row(p, b, si, j, hk, 1) : nullptr;
        rv[u] = rv_ptr ? *reinterpret_cast<const uint4*>(rv_ptr + cg * 8) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      add_units(raw[u].x, hi[0], lo[0], hi[1], lo[1]);
      add_units(raw[u].y, hi[2], lo[2], hi[3], lo[3]);
      add_units(raw[u].z, hi[4], lo[4], hi[5], lo[5]);
      add_units(raw[u].w, hi[6], lo[6], hi[7], lo[7]);
      if (want_v) {
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&rv[u]);
#pragma unroll
        for (int e = 0; e < 8; ++e) vmax[e] = fmaxf(vmax[e], fabsf(__bfloat162float(h[e])));
      }
    }
  }
  // |hi| <= 16 * 2^21 and |lo| <= 16 * 2^20 per lane: no int32 overflow
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    s_part[kl][cg * 8 + e] = static_cast<long long>(hi[e]) * (1ll << 21) + lo[e];
    s_vmax[kl][cg * 8 + e] = vmax[e];
  }
  __syncthreads();
  const size_t base = (static_cast<size_t>(b) * p.n_heads_kv + hk) * p.head_dim;
  if (threadIdx.x < 128) {
    long long t = 0;
    float vm = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      t += s_part[k][threadIdx.x];
      vm = fmaxf(vm, s_vmax[k][threadIdx.x]);
    }
    atomicAdd(reinterpret_cast<unsigned long long*>(p.sc.k_sum + base + threadIdx.x),
              static_cast<unsigned long long>(t));
    if (want_v) atomicMax(p.sc.v_amax + base + threadIdx.x, __float_as_uint(vm));
    __threadfence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned chunks = static_cast<unsigned>((L + kSumKeys - 1) / kSumKeys);
    s_last = atomicAdd(p.sc.k_cnt + static_cast<size_t>(b) * p.n_heads_kv + hk, 1u) == chunks - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x < 128) {
    const long long sum = __ldcg(p.sc.k_sum + base + threadIdx.x);
    p.sc.k_mean[base + threadIdx.x] =
        __double2float_rn(static_cast<double>(sum) * (1.0 / 4294967296.0) / static_cast<double>(L));
    if (want_v) {
      const float amax = __uint_as_float(__ldcg(p.sc.v_amax + base + threadIdx.x));
      p.v_scale[base + threadIdx.x] = e4m3_scale(amax);
      p.sc.v_inv[base + threadIdx.x] = e4m3_inv_scale(amax);
    }
  }
}

// grid (num_seqs * n_heads_kv, blocks per sequence), 256 threads: thread t
// quantises row t / 4 of the 64-key block, channels (t % 4) * 32 ... + 31.
__global__ void __launch_bounds__(256) k_quant_kernel(const QuantParams p) {
  grid_dep_launch();
  grid_dep_wait();  // the offsets are complete
  __shared__ float s_amax[8];
  __shared__ float s_mean[128];
  const int b = blockIdx.x / p.n_heads_kv, hk = blockIdx.x % p.n_heads_kv;
  const int blk = blockIdx.y;
  const int4 si = p.seq_info[b];
  if (si.y < 0) return;
  const int L = si.z;
  if (blk * kPage >= L) return;
  if (threadIdx.x < 128)
    s_mean[threadIdx.x] = p.sc.k_mean[(static_cast<size_t>(b) * p.n_heads_kv + hk) * p.head_dim + threadIdx.x];
  const int r = threadIdx.x >> 2, c0 = (threadIdx.x & 3) * 32;
  const int j = blk * kPage + r;
  const __nv_bfloat16* kr = j < L ? key_row(p, b, si, j, hk) : nullptr;
  uint4 raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    raw[i] = kr ? *reinterpret_cast<const uint4*>(kr + c0 + i * 8) : make_uint4(0, 0, 0, 0);
  __syncthreads();
  float x[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&raw[i]);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      x[i * 8 + e] = kr ? __fsub_rn(__bfloat162float(h[e]), s_mean[c0 + i * 8 + e]) : 0.f;
      amax = fmaxf(amax, fabsf(x[i * 8 + e]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) s_amax[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = s_amax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, s_amax[w]);
  const float inv = e4m3_inv_scale(amax);
  const size_t gblk = static_cast<size_t>(b) * p.nb_max + blk;
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const uint32_t lo = e4m3x2(__fmul_rn(x[i], inv), __fmul_rn(x[i + 1], inv));
    const uint32_t hi = e4m3x2(__fmul_rn(x[i + 2], inv), __fmul_rn(x[i + 3], inv));
    w[i / 4] = kr ? (lo | (hi << 16)) : 0u;
  }
  uint4* dst = reinterpret_cast<uint4*>(
      p.k8 + ((gblk * kPage + r) * p.n_heads_kv + hk) * p.head_dim + c0);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  if (threadIdx.x == 0) p.k_scale[gblk * p.n_heads_kv + hk] = e4m3_scale(amax);
}

// grid (num_seqs * n_heads_kv, 128-key tiles per sequence), 256 threads:
// thread t codes keys 8 (t % 16) ... + 7 of the tile at channels 8 (t / 16) ...
// + 7, packs the eight codes of each channel into 8 bytes of the transposed
// tile in shared memory ([channel][key]: 16 lanes fill one 128-byte channel
// row), and the CTA then writes the 16 KB tile out with 16-byte stores.
__global__ void __launch_bounds__(256) v_quant_kernel(const QuantParams p) {
  grid_dep_launch();
  grid_dep_wait();  // the V scales are complete
  __shared__ __align__(16) uint8_t s_t[128 * 128];
  const int b = blockIdx.x / p.n_heads_kv, hk = blockIdx.x % p.n_heads_kv;
  const int tile = blockIdx.y;
  const int4 si = p.seq_info[b];
  if (si.y < 0) return;
  const int L = si.z;
  if (tile * 128 >= L) return;
  const int kg = threadIdx.x & 15, cg = threadIdx.x >> 4;
  const size_t base = (static_cast<size_t>(b) * p.n_heads_kv + hk) * p.head_dim + cg * 8;
  const float4 i0 = *reinterpret_cast<const float4*>(p.sc.v_inv + base);
  const float4 i1 = *reinterpret_cast<const float4*>(p.sc.v_inv + base + 4);
  const float inv[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
  uint4 raw[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int j = tile * 128 + kg * 8 + u;
    const __nv_bfloat16* r = j < L ? kv_row(p, b, si, j, hk, 1) : nullptr;
    raw[u] = r ? *reinterpret_cast<const uint4*>(r + cg * 8) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      x[u] = __fmul_rn(__bfloat162float(reinterpret_cast<const __nv_bfloat16*>(&raw[u])[e]), inv[e]);
    const uint32_t w0 = e4m3x2(x[0], x[1]) | (e4m3x2(x[2], x[3]) << 16);
    const uint32_t w1 = e4m3x2(x[4], x[5]) | (e4m3x2(x[6], x[7]) << 16);
    *reinterpret_cast<uint2*>(s_t + (cg * 8 + e) * 128 + kg * 8) = make_uint2(w0, w1);
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(
      p.v8 + ((static_cast<size_t>(b) * (p.nb_max / 2) + tile) * p.n_heads_kv + hk) * (128 * 128));
  const uint4* src = reinterpret_cast<const uint4*>(s_t);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[threadIdx.x + i * 256] = src[threadIdx.x + i * 256];
}

// Query rows (token, head): eight lanes per row (lane holds 16 channels, two
// 16-byte loads), four rows per warp pass and two passes in flight. It needs
// nothing of the plan, but its completion is what the attention kernel waits
// for, so it waits for the K quantisation before it exits.
__global__ void __launch_bounds__(256) q_quant_kernel(const QuantParams p) {
  grid_dep_launch();
  const int lane = threadIdx.x & 31, g = lane >> 3, sub = lane & 7;
  const size_t rows = static_cast<size_t>(p.total_q) * p.n_heads_q;
  const size_t warps = static_cast<size_t>(gridDim.x) * (blockDim.x >> 5);
  for (size_t r0 = (static_cast<size_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 8; r0 < rows;
       r0 += warps * 8) {
    uint4 raw[2][2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const size_t row = r0 + u * 4 + g;
      const uint4* src = reinterpret_cast<const uint4*>(p.q + row * 128 + sub * 16);
      raw[u][0] = row < rows ? src[0] : make_uint4(0, 0, 0, 0);
      raw[u][1] = row < rows ? src[1] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const size_t row = r0 + u * 4 + g;
      const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&raw[u][0]);
      float x[16];
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        x[e] = __bfloat162float(h[e]);
        amax = fmaxf(amax, fabsf(x[e]));
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (row >= rows) continue;
      const float inv = e4m3_inv_scale(amax);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const uint32_t lo = e4m3x2(__fmul_rn(x[i], inv), __fmul_rn(x[i + 1], inv));
        const uint32_t hi = e4m3x2(__fmul_rn(x[i + 2], inv), __fmul_rn(x[i + 3], inv));
        w[i / 4] = lo | (hi << 16);
      }
      reinterpret_cast<uint4*>(p.q8 + row * 128)[sub] = make_uint4(w[0], w[1], w[2], w[3]);
      if (sub == 0) p.q_scale[row] = e4m3_scale(amax);
    }
  }
  grid_dep_wait();  // the K codes are complete before this grid is
}

}  // namespace

// After the plan (the zeroed part of the scratch cleared before it, in stream
// order): key sums, offsets and V scales, then K codes, V codes and Q codes as
// requested, each a dependent launch. The Q pass, when present, is last: its
// completion covers the others.
cudaError_t launch_quant(const QuantParams& p, int sms, cudaStream_t s) {
  cudaError_t e = launch_kernel(k_sum_kernel, dim3(p.num_seqs * p.n_heads_kv,
                                                   (p.nb_max * kPage + kSumKeys - 1) / kSumKeys),
                                256, 0, s, true, p);
  if (e == cudaSuccess && p.k8)
    e = launch_kernel(k_quant_kernel, dim3(p.num_seqs * p.n_heads_kv, p.nb_max), 256, 0, s, true, p);
  if (e == cudaSuccess && p.v8)
    e = launch_kernel(v_quant_kernel, dim3(p.num_seqs * p.n_heads_kv, p.nb_max / 2), 256, 0, s, true, p);
  if (e != cudaSuccess || !p.q8) return e;
  const size_t rows = static_cast<size_t>(p.total_q) * p.n_heads_q;
  const int blocks = static_cast<int>(std::min<size_t>((rows + 63) / 64, static_cast<size_t>(sms) * 8));
  return launch_kernel(q_quant_kernel, std::max(blocks, 1), 256, 0, s, true, p);
}

}  // namespace pattn
