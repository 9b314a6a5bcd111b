// decode.cu -- swap-AB paged decode attention for sm_103a (tcgen05 + TMA).
//
// For units whose packed query rows (query tokens x GQA group) fit in 16, the
// roles of the operands are swapped, as the trtllm-gen paged decode manifest's
// kernel ("...StaticSwapsAbForGen") does for generation:
//
//   S^T [128 keys x 16 rows] = K_tile [128 x D] . Q^T [D x 16]   (M = 128 keys, N = 16)
//   O^T [D x 16]            += V^T [D x 128]    . P^T [128 x 16]  (M = 128 d, N = 16)
//
// so the keys of a tile sit on the 128 TMEM lanes and each softmax thread owns
// ONE key: per tile it computes only as many exponentials as there are query
// rows, instead of 128 per row. The running max per query row needs a
// cross-thread reduction (warp shuffles, then four warps through shared
// memory); the running sum stays per thread and is reduced once per item.
//
// K and V tiles stream through one ring of R stages (R x 32 KB for D = 128,
// R x 64 KB for D = 256, about 192 KB in total), filled in the order
// K0 V0 K1 V1 ... by the load warp, which reads the block table 32 tiles at a
// time across its lanes (one page pair per lane) so that no TMA issue waits
// on a global load. The tail warp forwards every filled stage, zeroing V rows
// past the sequence end first (so 0 * NaN cannot reach O).
#include "kernels.cuh"
#include "merge.cuh"
#include "ptx.cuh"

namespace pattn {
namespace {

constexpr int kNQ = 16;   // packed query rows of a decode item (MMA N)
constexpr int kDBN = 128; // keys per tile (MMA M of S^T)

template <int D>
struct DCfg {
  static constexpr int kStage = kDBN * D * 2;              // one K or V tile
  static constexpr int kRing = D == 128 ? 6 : 3;            // stages
  static constexpr int kQBytes = kNQ * D * 2;
  static constexpr int kPBytes = kNQ * kDBN * 2;
  static constexpr int kOffRing = 0;
  static constexpr int kOffQ = kOffRing + kRing * kStage;
  static constexpr int kOffP = kOffQ + kQBytes;
  static constexpr int kOffRed = kOffP + 2 * kPBytes;       // 3 x 4 warps x 16 floats
  static constexpr int kOffBar = kOffRed + 3 * 4 * kNQ * 4;
  static constexpr int kOffMisc = kOffBar + 512;
  static constexpr int kSmem = kOffMisc + 64 + 1024;
  static constexpr int kDBlocks = D / 64;
  static constexpr int kHalves = D / 128;                  // M = 128 slices of O^T
  static constexpr int kColS = 0;                          // two S^T buffers of 16 columns
  static constexpr int kColO = 2 * kNQ;                    // kHalves x 16 columns
  static constexpr int kTmem = 64;
  static_assert(kColO + kHalves * kNQ <= kTmem, "TMEM");
  static_assert(kSmem <= 232448, "shared memory");
};

// P is double-buffered: p_full[b] / pv_done[b] complete once per use of P buffer b.
enum DBar { kDQFull = 0, kDQEmpty, kDSFull0, kDSFull1, kDSFree0, kDSFree1, kDPFull0, kDPFull1,
            kDPVDone0, kDPVDone1, kDDrain, kDRedMax0, kDRedMax1, kDRedSum, kDMerge0, kDMerge1,
            kDRingFull0 = 16,    // then ring full [R], ring ready [R], ring empty [R]
            kDDrainPV = 40 };    // the PV warp's drain (after the ring's 3 R <= 18)

struct SoftCtx {
  uint8_t* smem;
  uint32_t sBar, tmem, lane_base;
  int sw, t, lane;
  WaitCtl ctl;
  volatile int* merge_flag;  // shared: this CTA finished a split unit last
};

// One decode item on the softmax warpgroup. NR >= the item's packed query
// rows: only NR columns of S^T, P and O^T are touched. Returns false when a
// bounded wait gave up.
template <int D, int NR>
__device__ __forceinline__ bool softmax_item(const SoftCtx& x, const AttnParams& p, int4 iv,
                                             int4 si, uint32_t& n, uint32_t& itl, uint32_t& nsp) {
  using C = DCfg<D>;
  const unsigned full = 0xffffffffu;
  auto bar = [&](int i) { return x.sBar + 8u * static_cast<uint32_t>(i); };
  float* red = reinterpret_cast<float*>(x.smem + C::kOffRed);
  float* red_max = red;                 // [2][4][16]
  float* red_sum = red + 2 * 4 * kNQ;   // [4][16]
  const int G = p.group;
  const int hk = iv.y >> 16;
  const int kt0 = (iv.z >> 16) & 0xFFFF, kt1 = iv.z & 0xFFFF;
  const int q0 = si.x, ql = si.y, L = si.z;
  const int rows = ql * G;
  const int part = iv.w;  // first partial row of this split, -1 if not split
  const float c = p.scale_log2;
  const int t = x.t, lane = x.lane, sw = x.sw;
  int lim[NR];
  float m[NR], lp[NR];
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    const int tok = j / G;
    lim[j] = j < rows ? (p.causal ? min(L, L - ql + tok + 1) : L) : 0;
    m[j] = -INFINITY;
    lp[j] = 0.f;
  }
  for (int kt = kt0; kt < kt1; ++kt, ++n) {
    const uint32_t sb = n & 1u;
    const bool first = kt == kt0;
    if (!wait_warp(bar(kDSFull0 + sb), (n >> 1) & 1u, x.ctl)) return false;
    tc_fence_after();
    uint32_t sr[NR];
    tmem_ld(x.tmem + x.lane_base + C::kColS + sb * kNQ, sr);
    tmem_wait_ld();
    reg_fence(sr);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kDSFree0 + sb));

    const int key = kt * kDBN + t;
    float s[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) s[j] = key < lim[j] ? __uint_as_float(sr[j]) : -INFINITY;
    // tile max per query row: warp shuffles, then the four warps through shared memory
    float* rb = red_max + sb * (4 * kNQ);
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      float v = s[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(full, v, o));
      if (lane == 0) rb[sw * kNQ + j] = v;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kDRedMax0 + sb));
    if (!wait_warp(bar(kDRedMax0 + sb), (n >> 1) & 1u, x.ctl)) return false;
    bool any_need = false;
    float alpha[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      alpha[j] = 1.f;
      const float tm = fmaxf(fmaxf(rb[j], rb[kNQ + j]), fmaxf(rb[2 * kNQ + j], rb[3 * kNQ + j]));
      const float tms = tm == -INFINITY ? -INFINITY : tm * c;
      const float mn = fmaxf(m[j], tms);
      if (first) {
        m[j] = mn;
      } else if (mn > m[j] + 8.0f) {
        alpha[j] = ex2(m[j] - mn);
        m[j] = mn;
        any_need = true;
      }
    }
    if (any_need) {
      // rescale the O^T columns of the rows whose max grew, once the previous PV is done
      const uint32_t pm = n - 1;
      if (!wait_warp(bar(kDPVDone0 + (pm & 1u)), (pm >> 1) & 1u, x.ctl)) return false;
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < C::kHalves; ++h) {
        uint32_t o[NR];
        tmem_ld(x.tmem + x.lane_base + C::kColO + h * kNQ, o);
        tmem_wait_ld();
        reg_fence(o);
#pragma unroll
        for (int j = 0; j < NR; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha[j]);
        tmem_st(x.tmem + x.lane_base + C::kColO + h * kNQ, o);
      }
      tmem_wait_st();
#pragma unroll
      for (int j = 0; j < NR; ++j) lp[j] *= alpha[j];
    }
    float pr[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      const float mref = m[j] == -INFINITY ? 0.f : m[j];
      pr[j] = s[j] == -INFINITY ? 0.f : ex2(fmaf(s[j], c, -mref));
      lp[j] += pr[j];
    }
    // P buffer sb was last read by the PV of tile n - 2
    if (n >= 2) {
      const uint32_t pm = n - 2;
      if (!wait_warp(bar(kDPVDone0 + (pm & 1u)), (pm >> 1) & 1u, x.ctl)) return false;
    }
    // P [16 rows][128 keys], K-major B operand: key block t/64, 128-byte rows
    {
      uint8_t* pb = x.smem + C::kOffP + sb * C::kPBytes + (t >> 6) * (kNQ * 128);
      const int k = t & 63;
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        __nv_bfloat16 h = __float2bfloat16_rn(pr[j]);
        *reinterpret_cast<__nv_bfloat16*>(pb + j * 128 + (((k >> 3) ^ (j & 7)) << 4) + (k & 7) * 2) = h;
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kDPFull0 + sb));
  }
  // ------------------------------------------------------------ epilogue
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    float v = lp[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(full, v, o);
    if (lane == 0) red_sum[sw * kNQ + j] = v;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(bar(kDRedSum));
  if (!wait_warp(bar(kDRedSum), itl & 1u, x.ctl)) return false;
  ++itl;
  float inv[NR];
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    const float l = (red_sum[j] + red_sum[kNQ + j]) + (red_sum[2 * kNQ + j] + red_sum[3 * kNQ + j]);
    inv[j] = l > 0.f ? 1.f / l : 0.f;
    if (part >= 0 && t == 0 && j < rows) p.part_ml[part + j] = make_float2(l > 0.f ? m[j] : -INFINITY, l);
  }
  const uint32_t pm = n - 1;
  if (!wait_warp(bar(kDPVDone0 + (pm & 1u)), (pm >> 1) & 1u, x.ctl)) return false;
  tc_fence_after();
#pragma unroll
  for (int h = 0; h < C::kHalves; ++h) {
    uint32_t o[NR];
    tmem_ld(x.tmem + x.lane_base + C::kColO + h * kNQ, o);
    tmem_wait_ld();
    reg_fence(o);
    const int d = h * 128 + t;
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      if (j >= rows) continue;
      const float v = __uint_as_float(o[j]) * inv[j];
      if (part < 0) {
        const int tok = j / G, g = j - tok * G;
        p.out[(static_cast<size_t>(q0 + tok) * p.n_heads_q + hk * G + g) * D + d] = __float2bfloat16_rn(v);
      } else {
        p.part_o[static_cast<size_t>(part + j) * D + d] = v;
      }
    }
  }
  tc_fence_before();
  if (part >= 0) {
    // hand the written partials to the merge warp (which took the previous split item)
    if (!wait_warp(bar(kDMerge1), (nsp & 1u) ^ 1u, x.ctl)) return false;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kDMerge0));
    ++nsp;
  }
  return true;
}


template <int D>
__global__ void __launch_bounds__(kThreads, 1)
decode_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kv,
              const AttnParams p) {
  using C = DCfg<D>;
  constexpr int R = C::kRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t sRing = s_base + C::kOffRing;
  const uint32_t sQ = s_base + C::kOffQ;
  const uint32_t sP = s_base + C::kOffP;
  const uint32_t sBar = s_base + C::kOffBar;
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);
  uint8_t* misc = smem + C::kOffMisc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 16);
  // drains wait on their own control word, which nothing sets: after an abort
  // they still wait (bounded) for every copy and MMA in flight to complete
  volatile int* never_abort = reinterpret_cast<volatile int*>(misc + 20);
  auto bar = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };
  auto ring_full = [&](uint32_t s) { return bar(kDRingFull0 + static_cast<int>(s)); };
  auto ring_ready = [&](uint32_t s) { return bar(kDRingFull0 + R + static_cast<int>(s)); };
  auto ring_empty = [&](uint32_t s) { return bar(kDRingFull0 + 2 * R + static_cast<int>(s)); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtl ctl{abort_flag, p.err};
  const WaitCtl drain_ctl{never_abort, p.err};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *never_abort = 0;
    mbar_init(bar(kDQFull), 1);
    mbar_init(bar(kDQEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kDSFull0 + s), 1);
      mbar_init(bar(kDSFree0 + s), 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kDPFull0 + s), 4);
      mbar_init(bar(kDPVDone0 + s), 1);
    }
    mbar_init(bar(kDDrain), 1);
    mbar_init(bar(kDDrainPV), 1);
    mbar_init(bar(kDRedMax0), 4);
    mbar_init(bar(kDRedMax1), 4);
    mbar_init(bar(kDRedSum), 4);
    mbar_init(bar(kDMerge0), 4);  // a split item's partial rows are written (softmax warps)
    mbar_init(bar(kDMerge1), 1);  // the merge warp has taken that item
    for (int s = 0; s < R; ++s) {
      mbar_init(ring_full(s), 1);
      mbar_init(ring_ready(s), 1);
      mbar_init(ring_empty(s), 1);
    }
    mbar_init_fence();
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_kv);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmem);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();    // the plan is complete from here on
  // tell the prefill kernel so (it may start on this rather than on this grid)
  if (p.go && blockIdx.x == 0 && threadIdx.x == 0) st_release_gpu(p.go, 1);
  grid_dep_launch();  // the prefill kernel may take SMs as this grid's CTAs leave

  const int n_items = p.hdr[kHdrDecItems];
  const int G = p.group;
  const int Tq = p.tokens_per_tile;  // query tokens per decode item (kNQ / G)
  const unsigned full = 0xffffffffu;

  if (warp == 0) {
    // ------------------------------------------------------------ load warp (all lanes)
    uint32_t f = 0, itl = 0, qf = 0;  // ring fills, items, Q fills
    bool ok = true;
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    for (int kq = 0, idx = blockIdx.x; idx < n_items && ok;
         idx = cta_item(++kq, blockIdx.x, gridDim.x), ++itl) {
      const int4 iv = p.items[idx];
      const int b = iv.x & kSeqMask, hk = iv.y >> 16;
      const int kt0 = (iv.z >> 16) & 0xFFFF, kt1 = iv.z & 0xFFFF;
      const int4 si = p.seq_info[b];
      const int q0 = si.x, L = si.z, kv0 = si.w;
      if (lane == 0) {
        ok = wait_one(bar(kDQEmpty), (itl & 1u) ^ 1u, ctl);
        if (ok) {
          mbar_arrive_expect_tx(bar(kDQFull), static_cast<uint32_t>(C::kDBlocks * 128 * G * Tq));
          for (int c = 0; c < C::kDBlocks; ++c)
            tma_load_4d(sQ + c * (kNQ * 128), &tmap_q, bar(kDQFull), c * 64, 0, hk, q0, pol_q);
          ++qf;
        }
      }
      ok = __shfl_sync(full, ok, 0);
      const int ntiles = kt1 - kt0;
      for (int t0 = 0; t0 < ntiles && ok; t0 += 32) {
        // lane l fetches the two pages of tile t0 + l
        int pg0 = -1, pg1 = -1;
        const int tl = t0 + lane;
        if (tl < ntiles) {
          const int key = (kt0 + tl) * kDBN;
          if (p.paged) {
            const int32_t* row = p.block_table + static_cast<size_t>(b) * p.bt_stride;
            if (key < L) pg0 = row[key / kPage];
            if (key + kPage < L) pg1 = row[key / kPage + 1];
            if (pg0 >= p.num_pages || (key < L && pg0 < 0)) { atomicOr(p.err, kErrBadInput); pg0 = -1; }
            if (pg1 >= p.num_pages || (key + kPage < L && pg1 < 0)) { atomicOr(p.err, kErrBadInput); pg1 = -1; }
          } else {
            if (key < L) pg0 = kv0 + key;
            if (key + kPage < L) pg1 = kv0 + key + kPage;
          }
        }
        const int nb = min(32, ntiles - t0);
        for (int i = 0; i < nb; ++i) {
          const int a0 = __shfl_sync(full, pg0, i);
          const int a1 = __shfl_sync(full, pg1, i);
          if (lane == 0) {
            const int nload = (a0 >= 0) + (a1 >= 0);
            const uint32_t bytes = static_cast<uint32_t>(nload * C::kDBlocks * kPage * 128);
            for (int kind = 0; kind < 2 && ok; ++kind, ++f) {
              const uint32_t s = f % R, ph = (f / R) & 1u;
              ok = wait_one(ring_empty(s), ph ^ 1u, ctl);
              if (!ok) break;
              mbar_arrive_expect_tx(ring_full(s), bytes);
              const uint32_t dst0 = sRing + s * C::kStage;
              for (int pg = 0; pg < 2; ++pg) {
                const int a = pg ? a1 : a0;
                if (a < 0) continue;
                for (int c = 0; c < C::kDBlocks; ++c) {
                  const uint32_t dst = dst0 + c * (kDBN * 128) + pg * (kPage * 128);
                  if (p.paged)
                    tma_load_4d(dst, &tmap_kv, ring_full(s), c * 64, 0, hk, 2 * a + kind, pol_kv);
                  else
                    tma_load_4d(dst, &tmap_kv, ring_full(s), c * 64, hk, a, kind, pol_kv);
                }
              }
            }
          }
          ok = __shfl_sync(full, ok, 0);
          if (!ok) break;
        }
      }
    }
    // drain: the last fill of every stage, and the last Q fill, have landed
    if (lane == 0) {
      for (uint32_t s = 0; s < static_cast<uint32_t>(R); ++s) {
        if (f <= s) continue;
        const uint32_t last = ((f - 1 - s) / R) * R + s;
        wait_one(ring_full(s), (last / R) & 1u, drain_ctl);
      }
      if (qf > 0) wait_one(bar(kDQFull), (qf - 1) & 1u, drain_ctl);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK MMA warp
    // S^T = K Q^T for every tile, issued by one thread; the PV MMAs come from
    // warp 8, so that a PV waiting for its P never holds up the next QK (and
    // each V stage is released as soon as its PV is done)
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kNQ, false, false);
      const SmemDesc dring_k = sw128_desc_split(sRing, 16, 1024);          // K tiles, K-major
      const SmemDesc dq = sw128_desc_split(sQ, 16, 1024);
      uint32_t n = 0, itl = 0;
      bool ok = true;
      // failure-detection self-test: the first CTA's MMA thread first waits for a
      // phase that nothing completes before the drain below, so the wait runs
      // out and every role of the CTA takes its abort path
      if (p.selftest_abort && blockIdx.x == 0 && n_items > 0) ok = wait_one(bar(kDDrain), 0, ctl);
      for (int kq = 0, idx = blockIdx.x; idx < n_items && ok;
         idx = cta_item(++kq, blockIdx.x, gridDim.x), ++itl) {
        const int4 iv = p.items[idx];
        const int kt0 = (iv.z >> 16) & 0xFFFF, kt1 = iv.z & 0xFFFF;
        if (!(ok = wait_one(bar(kDQFull), itl & 1u, ctl))) break;
        tc_fence_after();
        for (int kt = kt0; kt < kt1; ++kt, ++n) {
          const uint32_t fk = 2 * n, s = fk % R, ph = (fk / R) & 1u;
          const uint32_t sb = n & 1u;
          if (!(ok = wait_one(ring_ready(s), ph, ctl))) break;
          if (!(ok = wait_one(bar(kDSFree0 + sb), ((n >> 1) & 1u) ^ 1u, ctl))) break;
          tc_fence_after();
          const uint32_t k_lo = desc_lo_at(dring_k, s * C::kStage);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t a_lo = k_lo + (((kk >> 2) * (kDBN * 128) + (kk & 3) * 32) >> 4);
            const uint32_t b_lo = dq.lo + (((kk >> 2) * (kNQ * 128) + (kk & 3) * 32) >> 4);
            umma_f16_ss(tmem + C::kColS + sb * kNQ, a_lo, dring_k.hi, b_lo, dq.hi, idesc_qk,
                        kk > 0 ? 1u : 0u);
          }
          umma_commit(ring_empty(s));
          umma_commit(bar(kDSFull0 + sb));
        }
        if (!ok) break;
        umma_commit(bar(kDQEmpty));  // the item's last QK has read Q
      }
      umma_commit(bar(kDDrain));
      wait_one(bar(kDDrain), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ ring forwarder / V tail fix
    uint32_t n = 0;
    bool ok = true;
    for (int kq = 0, idx = blockIdx.x; idx < n_items && ok; idx = cta_item(++kq, blockIdx.x, gridDim.x)) {
      const int4 iv = p.items[idx];
      const int kt0 = (iv.z >> 16) & 0xFFFF, kt1 = iv.z & 0xFFFF;
      const int L = p.seq_info[iv.x & kSeqMask].z;
      for (int kt = kt0; kt < kt1; ++kt, ++n) {
        for (uint32_t kind = 0; kind < 2; ++kind) {
          const uint32_t fi = 2 * n + kind, s = fi % R, ph = (fi / R) & 1u;
          if (!(ok = wait_warp(ring_full(s), ph, ctl))) break;
          const int live = L - kt * kDBN;
          if (kind == 1 && live < kDBN) {
            uint8_t* v0 = smem + C::kOffRing + s * C::kStage;
            const int chunks = (kDBN - live) * 8;
            for (int c = 0; c < C::kDBlocks; ++c) {
              uint4* blk = reinterpret_cast<uint4*>(v0 + c * (kDBN * 128) + live * 128);
              for (int i = lane; i < chunks; i += 32) blk[i] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(ring_ready(s));
        }
        if (!ok) break;
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ split merge warp
    // For every split item: once its partials are written, count it; the CTA
    // that finished the unit's last split merges the unit here, off the softmax
    // warps' path.
    uint32_t nsp = 0;
    bool ok = true;
    for (int kq = 0, idx = blockIdx.x; idx < n_items && ok; idx = cta_item(++kq, blockIdx.x, gridDim.x)) {
      const int4 iv = p.items[idx];
      if (iv.w < 0) continue;
      if (!(ok = wait_warp(bar(kDMerge0), nsp & 1u, ctl))) break;
      const int4 sp = p.seq_plan[iv.x & kSeqMask];
      int last = 0;
      if (lane == 0) {
        __threadfence();
        last = atomicAdd(&p.unit_cnt[sp.w + (iv.y >> 16)], 1) == sp.z - 1;
        if (last) __threadfence();
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kDMerge1));
      ++nsp;
      if (last) {
        const int4 si = p.seq_info[iv.x & kSeqMask];
        const int rows = si.y * G;
        merge_unit<D, D == 256 ? 2 : 4>(p, si.x, iv.y >> 16, sp.z, iv.w - (iv.x >> kSeqBits) * rows, rows, 0, 1);
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ PV MMA warp
    // O^T += V^T P^T for every tile, one thread, as soon as the tile's P is
    // written and its V stage forwarded; the commit releases that V stage
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, kNQ, true, false);
      const SmemDesc dring_v = sw128_desc_split(sRing, kDBN * 128, 1024);  // V tiles, MN-major
      const SmemDesc dp = sw128_desc_split(sP, 16, 1024);
      uint32_t n = 0;
      bool ok = true;
      for (int kq = 0, idx = blockIdx.x; idx < n_items && ok; idx = cta_item(++kq, blockIdx.x, gridDim.x)) {
        const int4 iv = p.items[idx];
        const int kt0 = (iv.z >> 16) & 0xFFFF, kt1 = iv.z & 0xFFFF;
        for (int kt = kt0; kt < kt1; ++kt, ++n) {
          const uint32_t fv = 2 * n + 1, s = fv % R, ph = (fv / R) & 1u;
          if (!(ok = wait_one(bar(kDPFull0 + (n & 1u)), (n >> 1) & 1u, ctl))) break;
          if (!(ok = wait_one(ring_ready(s), ph, ctl))) break;
          tc_fence_after();
          const uint32_t v_lo = desc_lo_at(dring_v, s * C::kStage);
          const uint32_t p_lo = desc_lo_at(dp, (n & 1u) * C::kPBytes);
          const bool first = kt == kt0;
#pragma unroll
          for (int kk = 0; kk < kDBN / 16; ++kk) {
            const uint32_t b_lo = p_lo + (((kk >> 2) * (kNQ * 128) + (kk & 3) * 32) >> 4);
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) {
              const uint32_t a_lo = v_lo + (((2 * h) * (kDBN * 128) + kk * (16 * 128)) >> 4);
              umma_f16_ss(tmem + C::kColO + h * kNQ, a_lo, dring_v.hi, b_lo, dp.hi, idesc_pv,
                          (first && kk == 0) ? 0u : 1u);
            }
          }
          umma_commit(ring_empty(s));
          umma_commit(bar(kDPVDone0 + (n & 1u)));
        }
      }
      umma_commit(bar(kDDrainPV));
      wait_one(bar(kDDrainPV), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax: one key per thread
    SoftCtx x;
    x.smem = smem;
    x.sBar = sBar;
    x.sw = warp - 4;
    x.t = threadIdx.x - 128;
    x.lane = lane;
    x.lane_base = static_cast<uint32_t>(x.sw * 32) << 16;
    x.tmem = tmem;
    x.ctl = ctl;
    x.merge_flag = reinterpret_cast<volatile int*>(misc + 32);
    uint32_t n = 0, itl = 0, nsp = 0;
    bool ok = true;
    for (int kq = 0, idx = blockIdx.x; idx < n_items && ok; idx = cta_item(++kq, blockIdx.x, gridDim.x)) {
      const int4 iv = p.items[idx];
      const int4 si = p.seq_info[iv.x & kSeqMask];
      const int rows = si.y * G;
      if (rows <= 4)
        ok = softmax_item<D, 4>(x, p, iv, si, n, itl, nsp);
      else if (rows <= 8)
        ok = softmax_item<D, 8>(x, p, iv, si, n, itl, nsp);
      else
        ok = softmax_item<D, 16>(x, p, iv, si, n, itl, nsp);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmem);
}

}  // namespace

size_t decode_smem_bytes(int head_dim) {
  return head_dim == 128 ? static_cast<size_t>(DCfg<128>::kSmem) : static_cast<size_t>(DCfg<256>::kSmem);
}

cudaError_t decode_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DCfg<128>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              DCfg<256>::kSmem);
}

cudaError_t launch_decode(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tkv,
                          int head_dim, int grid, cudaStream_t s, bool dependent) {
  if (head_dim == 128)
    return launch_kernel(decode_kernel<128>, grid, kThreads, DCfg<128>::kSmem, s, dependent, tq, tkv, p);
  return launch_kernel(decode_kernel<256>, grid, kThreads, DCfg<256>::kSmem, s, dependent, tq, tkv, p);
}

}  // namespace pattn
