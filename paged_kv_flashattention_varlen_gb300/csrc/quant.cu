// quant.cu -- the preparation phases of the quantised-QK variant (the GB10
// "sage2" benchmark page: k_mean_and_smoothing_preparation,
// q_int8_quantization, k_int8_subtract_mean_quantization), with fp8 e4m3 codes
// in place of int8: on sm_103a the e4m3 tensor-core rate is twice the bf16 one
// and the int8 rate is far below it.
//
//   * k_sum_kernel: per (sequence, KV head, channel), the sum of the sequence's
//     keys in float64. Each CTA adds up 1024 keys and adds its partial sums
//     into the total with float64 atomics. Sums of bf16 values are exact in
//     float64 at these lengths, so the order does not matter.
//   * k_quant_kernel: per (sequence, 64-key block, KV head): the mean (sum / L
//     in float64, rounded to fp32), x = k - mean in fp32, scale = amax / 448
//     (IEEE division; 1 when amax = 0), code = e4m3 round-to-nearest-even of
//     x / scale (IEEE division), saturated. Rows past L are zero codes.
//   * q_quant_kernel: per query row (token, head): scale = amax / 448 and codes
//     as above.
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

constexpr int kSumKeys = 1024;  // keys per k_sum CTA
constexpr float kE4m3Max = 448.0f;

__device__ __forceinline__ float e4m3_scale(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
}

// Two fp32 values -> two e4m3 bytes (first value in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Pointer to key row j of sequence b, KV head hk (nullptr if its page is not
// a pool page; the plan has then rejected the sequence already).
__device__ __forceinline__ const __nv_bfloat16* key_row(const QuantParams& p, int b, int4 si, int j, int hk) {
  const size_t row = static_cast<size_t>(p.n_heads_kv) * p.head_dim;
  if (p.block_table) {
    const int page = p.block_table[static_cast<size_t>(b) * p.bt_stride + j / kPage];
    if (page < 0 || page >= p.num_pages) return nullptr;
    return p.kv_pool + (static_cast<size_t>(page) * 2 * kPage + (j % kPage)) * row + static_cast<size_t>(hk) * p.head_dim;
  }
  return p.kv_pool + (static_cast<size_t>(si.w) + j) * row + static_cast<size_t>(hk) * p.head_dim;
}

// grid (num_seqs * n_heads_kv, key chunks), block head_dim threads: thread d
// sums channel d of kSumKeys keys.
__global__ void __launch_bounds__(128) k_sum_kernel(const QuantParams p) {
  grid_dep_launch();
  grid_dep_wait();  // the plan is complete
  const int b = blockIdx.x / p.n_heads_kv, hk = blockIdx.x % p.n_heads_kv;
  const int4 si = p.seq_info[b];
  if (si.y < 0) return;
  const int L = si.z;
  const int j0 = blockIdx.y * kSumKeys, j1 = min(L, j0 + kSumKeys);
  if (j0 >= j1) return;
  const int d = threadIdx.x;
  double acc[4] = {0.0, 0.0, 0.0, 0.0};
  int j = j0;
  for (; j + 4 <= j1; j += 4) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const __nv_bfloat16* r = key_row(p, b, si, j + u, hk);
      v[u] = r ? __bfloat162float(r[d]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] += static_cast<double>(v[u]);
  }
  for (; j < j1; ++j) {
    const __nv_bfloat16* r = key_row(p, b, si, j, hk);
    acc[0] += r ? static_cast<double>(__bfloat162float(r[d])) : 0.0;
  }
  atomicAdd(p.k_sum + (static_cast<size_t>(b) * p.n_heads_kv + hk) * p.head_dim + d,
            (acc[0] + acc[1]) + (acc[2] + acc[3]));
}

// grid (num_seqs * n_heads_kv, blocks per sequence), 256 threads: thread t
// quantises row t / 4 of the 64-key block, channels (t % 4) * 32 ... + 31.
__global__ void __launch_bounds__(256) k_quant_kernel(const QuantParams p) {
  grid_dep_launch();
  grid_dep_wait();  // the key sums are complete
  __shared__ float s_amax[8];
  const int b = blockIdx.x / p.n_heads_kv, hk = blockIdx.x % p.n_heads_kv;
  const int blk = blockIdx.y;
  const int4 si = p.seq_info[b];
  if (si.y < 0) return;
  const int L = si.z;
  if (blk * kPage >= L) return;
  const int r = threadIdx.x >> 2, c0 = (threadIdx.x & 3) * 32;
  const int j = blk * kPage + r;
  const double* sum = p.k_sum + (static_cast<size_t>(b) * p.n_heads_kv + hk) * p.head_dim + c0;
  float x[32];
  float amax = 0.f;
  const __nv_bfloat16* kr = j < L ? key_row(p, b, si, j, hk) : nullptr;
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (kr) raw = *reinterpret_cast<const uint4*>(kr + c0 + i);
    const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float mean = __double2float_rn(sum[i + e] / static_cast<double>(L));
      x[i + e] = kr ? __fsub_rn(__bfloat162float(h[e]), mean) : 0.f;
      amax = fmaxf(amax, fabsf(x[i + e]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) s_amax[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = s_amax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, s_amax[w]);
  const float scale = e4m3_scale(amax);
  const size_t gblk = static_cast<size_t>(b) * p.nb_max + blk;
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const uint32_t lo = e4m3x2(__fdiv_rn(x[i], scale), __fdiv_rn(x[i + 1], scale));
    const uint32_t hi = e4m3x2(__fdiv_rn(x[i + 2], scale), __fdiv_rn(x[i + 3], scale));
    w[i / 4] = kr ? (lo | (hi << 16)) : 0u;
  }
  uint4* dst = reinterpret_cast<uint4*>(
      p.k8 + ((gblk * kPage + r) * p.n_heads_kv + hk) * p.head_dim + c0);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  if (threadIdx.x == 0) p.k_scale[gblk * p.n_heads_kv + hk] = scale;
}

// One warp per query row (token, head), lane l holding channels 4l ... 4l + 3.
// It needs nothing of the plan, but its completion is what the attention kernel
// waits for, so it waits for the K quantisation before it exits.
__global__ void __launch_bounds__(256) q_quant_kernel(const QuantParams p) {
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const size_t rows = static_cast<size_t>(p.total_q) * p.n_heads_q;
  const size_t warps = static_cast<size_t>(gridDim.x) * (blockDim.x >> 5);
  for (size_t row = static_cast<size_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const uint2 raw = *reinterpret_cast<const uint2*>(p.q + row * p.head_dim + lane * 4);
    const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&raw);
    float x[4];
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] = __bfloat162float(h[e]);
      amax = fmaxf(amax, fabsf(x[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = e4m3_scale(amax);
    const uint32_t lo = e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale));
    const uint32_t hi = e4m3x2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale));
    reinterpret_cast<uint32_t*>(p.q8 + row * p.head_dim)[lane] = lo | (hi << 16);
    if (lane == 0) p.q_scale[row] = scale;
  }
  grid_dep_wait();  // the K codes are complete before this grid is
}

}  // namespace

// After the plan (k_sum zeroed before it, in stream order): key sums, K codes,
// Q codes, each a dependent launch.
cudaError_t launch_quant_qk(const QuantParams& p, int sms, cudaStream_t s) {
  cudaError_t e = launch_kernel(k_sum_kernel, dim3(p.num_seqs * p.n_heads_kv,
                                                   (p.nb_max * kPage + kSumKeys - 1) / kSumKeys),
                                128, 0, s, true, p);
  if (e != cudaSuccess) return e;
  e = launch_kernel(k_quant_kernel, dim3(p.num_seqs * p.n_heads_kv, p.nb_max), 256, 0, s, true, p);
  if (e != cudaSuccess) return e;
  const size_t rows = static_cast<size_t>(p.total_q) * p.n_heads_q;
  const int blocks = static_cast<int>(std::min<size_t>((rows + 7) / 8, static_cast<size_t>(sms) * 16));
  return launch_kernel(q_quant_kernel, std::max(blocks, 1), 256, 0, s, true, p);
}

}  // namespace pattn
