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
// Warp w of nw warps takes rows w, w + nw, ...; each lane D / 32 columns.
template <int D>
__device__ __forceinline__ void merge_unit(const AttnParams& p, int q0, int hk, int S, int base,
                                           int rows, int w, int nw) {
  const int lane = threadIdx.x & 31;
  constexpr int kPer = D / 32;
  const int G = p.group;
  for (int r = w; r < rows; r += nw) {
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, __ldcg(&p.part_ml[base + s * rows + r].x));
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < S; ++s) {
        const float2 ml = __ldcg(&p.part_ml[base + s * rows + r]);
        if (ml.y <= 0.f) continue;
        const float wt = ml.y * ex2(ml.x - M);
        den += wt;
        const float4* o = reinterpret_cast<const float4*>(
            p.part_o + static_cast<size_t>(base + s * rows + r) * D + lane * kPer);
#pragma unroll
        for (int e = 0; e < kPer / 4; ++e) {
          const float4 v = __ldcg(o + e);
          acc[4 * e] += wt * v.x;
          acc[4 * e + 1] += wt * v.y;
          acc[4 * e + 2] += wt * v.z;
          acc[4 * e + 3] += wt * v.w;
        }
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int tok = q0 + r / G;
    const int h = hk * G + r % G;
    __nv_bfloat16* dst = p.out + (static_cast<size_t>(tok) * p.n_heads_q + h) * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; e += 2)
      *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  }
}

}  // namespace pattn
