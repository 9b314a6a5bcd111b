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
// Warp w of nw warps takes rows w, w + nw, ...; each lane D / 32 columns. The
// S <= 64 splits' (m, l) are loaded at once (split s in lane s % 32, second
// slot for s >= 32) and reduced with shuffles; the partial O rows are then
// loaded four splits at a time, so that a row costs a few L2 round trips
// rather than two per split.
template <int D>
__device__ __forceinline__ void merge_unit(const AttnParams& p, int q0, int hk, int S, int base,
                                           int rows, int w, int nw) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  constexpr int kPer = D / 32;
  const int G = p.group;
  for (int r = w; r < rows; r += nw) {
    float2 a = make_float2(-INFINITY, 0.f), b = make_float2(-INFINITY, 0.f);
    if (lane < S) a = __ldcg(&p.part_ml[base + lane * rows + r]);
    if (lane + 32 < S) b = __ldcg(&p.part_ml[base + (lane + 32) * rows + r]);
    float M = fmaxf(a.x, b.x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(full, M, o));
    // weight of each split (0 for a split that saw no key)
    const float wa = (M != -INFINITY && a.y > 0.f) ? a.y * ex2(a.x - M) : 0.f;
    const float wb = (M != -INFINITY && b.y > 0.f) ? b.y * ex2(b.x - M) : 0.f;
    float den = wa + wb;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(full, den, o);
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    for (int s0 = 0; s0 < S; s0 += 4) {
      float4 v[4][kPer / 4];
      float wt[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int s = s0 + u;
        const float ws = __shfl_sync(full, s < 32 ? wa : wb, s & 31);
        wt[u] = s < S ? ws : 0.f;
        const float4* o = reinterpret_cast<const float4*>(
            p.part_o + static_cast<size_t>(base + min(s, S - 1) * rows + r) * D + lane * kPer);
#pragma unroll
        for (int e = 0; e < kPer / 4; ++e) v[u][e] = wt[u] > 0.f ? __ldcg(o + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < kPer / 4; ++e) {
          acc[4 * e] += wt[u] * v[u][e].x;
          acc[4 * e + 1] += wt[u] * v[u][e].y;
          acc[4 * e + 2] += wt[u] * v[u][e].z;
          acc[4 * e + 3] += wt[u] * v[u][e].w;
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
