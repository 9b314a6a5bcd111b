// merge.cuh -- in-kernel merge of split-KV partials (the decode manifest's
// "MultiCtasKv" reduction: its "counter" scratch counts finished splits, the
// "partial" and "stats" scratch hold each split's O and (max, sum)).
//
// Every split item writes its normalised partial O_s and (m_s, l_s), fences,
// and bumps the unit's counter; the CTA that finishes last merges:
//   M = max_s m_s,  w_s = l_s * 2^(m_s - M),  O = sum_s w_s O_s / sum_s w_s
// (m in log2 units; splits with l_s = 0 saw no key and weigh nothing).
#pragma once
#include "kernels.cuh"
#include "ptx.cuh"

namespace pattn {

// Rows r < rows of unit (q0, hk): split s of row r is at partial row base + s * rows.
// Warp w of nw warps takes rows in rounds of kRB (w, w + nw, ...; kRB rows
// loads in flight at once: more rows per round cost registers); each lane
// holds D / 32 columns. A round issues, before using any of them, the loads of
// its rows' split statistics (split s in lane s % 32, a second slot for
// s >= 32) and of the first four splits' partial O rows (every split writes
// all rows of its unit, finite, zero where it saw no key), so that it costs one
// L2 round trip; further splits load four at a time. A split's weight is
// applied with a select: one that saw no key adds exactly zero.
template <int D, int kRB>
__device__ __forceinline__ void merge_unit(const AttnParams& p, int q0, int hk, int S, int base,
                                           int rows, int w, int nw) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  constexpr int kPer = D / 32;
  constexpr int kV4 = kPer / 4;  // float4 loads per lane and partial row
  const int G = p.group;
  for (int r0 = w; r0 < rows; r0 += kRB * nw) {
    float2 a[kRB], b[kRB];
    float4 v[kRB][4][kV4];
#pragma unroll
    for (int j = 0; j < kRB; ++j) {
      const int r = r0 + j * nw;
      a[j] = make_float2(-INFINITY, 0.f);
      b[j] = make_float2(-INFINITY, 0.f);
      if (r < rows) {
        if (lane < S) a[j] = __ldcg(&p.part_ml[base + lane * rows + r]);
        if (lane + 32 < S) b[j] = __ldcg(&p.part_ml[base + (lane + 32) * rows + r]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4* o = reinterpret_cast<const float4*>(
            p.part_o + static_cast<size_t>(base + min(u, S - 1) * rows + min(r, rows - 1)) * D + lane * kPer);
#pragma unroll
        for (int e = 0; e < kV4; ++e)
          v[j][u][e] = (r < rows && u < S) ? __ldcg(o + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int j = 0; j < kRB; ++j) {
      const int r = r0 + j * nw;
      float M = fmaxf(a[j].x, b[j].x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(full, M, o));
      // weight of each split (0 for a split that saw no key)
      const float wa = (M != -INFINITY && a[j].y > 0.f) ? a[j].y * ex2(a[j].x - M) : 0.f;
      const float wb = (M != -INFINITY && b[j].y > 0.f) ? b[j].y * ex2(b[j].x - M) : 0.f;
      float den = wa + wb;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(full, den, o);
      float acc[kPer];
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
      for (int s0 = 0; s0 < S; s0 += 4) {
        float wt[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int s = s0 + u;
          const float ws = __shfl_sync(full, s < 32 ? wa : wb, s & 31);
          wt[u] = s < S ? ws : 0.f;
        }
        if (s0 > 0) {
          // splits s0 .. s0 + 3 (the first four came with the statistics)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float4* o = reinterpret_cast<const float4*>(
                p.part_o + static_cast<size_t>(base + min(s0 + u, S - 1) * rows + min(r, rows - 1)) * D +
                lane * kPer);
#pragma unroll
            for (int e = 0; e < kV4; ++e)
              v[j][u][e] = (r < rows && wt[u] > 0.f) ? __ldcg(o + e) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int e = 0; e < kV4; ++e) {
            const bool use = wt[u] > 0.f;
            acc[4 * e] += use ? wt[u] * v[j][u][e].x : 0.f;
            acc[4 * e + 1] += use ? wt[u] * v[j][u][e].y : 0.f;
            acc[4 * e + 2] += use ? wt[u] * v[j][u][e].z : 0.f;
            acc[4 * e + 3] += use ? wt[u] * v[j][u][e].w : 0.f;
          }
      }
      if (r >= rows) continue;
      const float inv = den > 0.f ? 1.f / den : 0.f;
      const int tok = q0 + r / G;
      const int h = hk * G + r % G;
      __nv_bfloat16* dst = p.out + (static_cast<size_t>(tok) * p.n_heads_q + h) * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 2)
        *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
    }
  }
}

}  // namespace pattn
