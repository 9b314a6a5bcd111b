// attn2q.cu -- head_dim-128 prefill with two q tiles per CTA, for sm_103a
// (tcgen05 + TMA).
//
// The two-Q-tile structure of the FlashAttention-4 SM100MHA2Q kernel doc (two
// Q tiles per CTA; softmax, correction, load and MMA warp roles; P taken from
// tensor memory by the second MMA) on the planner's paired items: an item is
// q tiles qt (A) and qt + 1 (B) of one (sequence, KV head) unit over the KV
// range of the later one, so every K and V tile is loaded once for both. The
// softmax of one q tile runs while the tensor pipe works on the other's MMAs.
//
// Warp roles (12 warps, one persistent CTA per SM):
//   * warp 0 TMA-loads both Q tiles of an item (GQA-packed: the G query heads
//     of one KV head for T = 128 / G tokens per tile) and the K tiles, warp 3
//     the V tiles, page by page through the pool's tensor map;
//   * warp 1 issues S_A = Q_A K^T and S_B = Q_B K^T (M 128, N 128, K 128) from
//     one thread;
//   * warp 2 zeroes V rows past the sequence end and issues O_A += P_A V and
//     O_B += P_B V (P from tensor memory) from one thread;
//   * warps 4-7 are the softmax of q tile A, warps 8-11 of q tile B: one query
//     row per thread, all 128 keys of a tile. P = 2^(S c - m) (the scale
//     folded into log2 e) is computed against the running max first; a row
//     sum of at most 2^8 bounds every p by 2^8, which is exactly when the
//     running max is kept, so the tile max is taken only otherwise (and on an
//     item's first tile). O is rescaled only when the row's max grows by more
//     than 2^8 (log2 units; exact, since O and the row sum share the stale
//     max). P (bf16 pairs) is written over the first half of S.
//
// Tensor memory (512 columns): O_A | O_B | S_A | S_B, P_X over the first 64
// columns of S_X. QK(X, n + 1) waits for PV(X, n), which reads P_X.
//
// At the end of an item each softmax warpgroup divides its O by its row sums
// and stores bf16 rows (a full q tile of an unsplit item through 32-column
// slices staged in shared memory and a tensor store), or, for a split item
// (a single q tile: only A has rows), writes the normalised partial O and
// (m, l), and the CTA that finishes the unit's last split merges it.
#include "kernels.cuh"
#include "merge.cuh"
#include "prefill.cuh"
#include "ptx.cuh"

namespace pattn {
namespace {

constexpr int kD2 = 128;          // head dim
constexpr int kBN2 = 128;         // keys per KV tile
constexpr int kThreads2 = 384;

struct Q2 {
  static constexpr int kQBytes = kBM * kD2 * 2;    // one q tile (32 KB)
  static constexpr int kStage = kBN2 * kD2 * 2;    // one K or V tile (32 KB)
  static constexpr int kStages = 2;
  static constexpr int kOffQ = 0;                  // Q_A | Q_B
  static constexpr int kOffK = kOffQ + 2 * kQBytes;
  static constexpr int kOffV = kOffK + kStages * kStage;
  // per softmax warpgroup: two buffers of one 32-column slice of its bf16 output
  // rows (64-byte rows, 64-byte swizzle) for the tensor store, so that a slice
  // is staged while the previous one is stored
  static constexpr int kOSlice = kBM * 64;
  static constexpr int kOffO = kOffV + kStages * kStage;
  static constexpr int kOffBar = kOffO + 4 * kOSlice;
  static constexpr int kOffMisc = kOffBar + 512;
  static constexpr int kSmem = kOffMisc + 128 + 1024;  // + alignment slack
  static constexpr int kColO = 0;                  // O_A | O_B
  static constexpr int kColS = 2 * kD2;            // S_A | S_B
  static_assert(kColS + 2 * kBN2 <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

// mbarrier slots. PV(X, n) done is tracked by two barriers per q tile by tile
// parity, so that no waiter can confuse a phase with the one two tiles later.
enum Bar2 {
  kQ2Full = 0, kQ2Empty,
  kK2Full0, kK2Full1, kK2Empty0, kK2Empty1,
  kV2Full0, kV2Full1,
  kS2Full0, kS2Full1,                 // S_X of the current tile written (X = A, B)
  kP2Full0, kP2Full1,                 // P_X written (4 warps each)
  kPV2A0, kPV2A1, kPV2B0, kPV2B1,     // PV(X, n) done, barrier 2 X + n % 2
  kDrain2, kDrainPV2, kMerge2A, kMerge2B,
  kSl2Full0, kSl2Full1, kSl2Full2, kSl2Full3,  // slice buffer 2 X + b staged by X's 4 warps
  kSl2Free0, kSl2Free1, kSl2Free2, kSl2Free3,  // the tensor store has read slice buffer 2 X + b
  kNumBars2
};
static_assert(kNumBars2 * 8 <= 512, "mbarrier area");

// Max of the first nv (of 32) scores of a chunk.
template <bool kMasked>
__device__ __forceinline__ float chunk_max(const uint32_t (&s)[32], int nv) {
  float acc[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) acc[u] = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (!kMasked || i < nv) acc[i & 7] = fmaxf(acc[i & 7], __uint_as_float(s[i]));
  return fmaxf(fmaxf(fmaxf(acc[0], acc[1]), fmaxf(acc[2], acc[3])),
               fmaxf(fmaxf(acc[4], acc[5]), fmaxf(acc[6], acc[7])));
}

// p_i = 2^(s_i c - m) for a 32-key chunk as 16 bf16 pairs; with kMasked only
// the first nv keys count. Returns the fp32 sum of the p_i (packed fp32x2 ops).
template <bool kMasked>
__device__ __forceinline__ float chunk_exp(const uint32_t (&s)[32], float c, float m, int nv,
                                           uint32_t (&pk)[16]) {
  const float2 c2 = make_float2(c, c);
  const float2 nm2 = make_float2(-m, -m);
  float2 acc[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) acc[u] = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[i]), __uint_as_float(s[i + 1])), c2, nm2);
    float p0 = ex2(x.x);
    float p1 = ex2(x.y);
    if constexpr (kMasked) {
      p0 = i < nv ? p0 : 0.f;
      p1 = i + 1 < nv ? p1 : 0.f;
    }
    acc[(i >> 1) & 3] = __fadd2_rn(acc[(i >> 1) & 3], make_float2(p0, p1));
    __nv_bfloat162 hh = __floats2bfloat162_rn(p0, p1);
    pk[i >> 1] = *reinterpret_cast<uint32_t*>(&hh);
  }
  const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  return a.x + a.y;
}

__global__ void __launch_bounds__(kThreads2, 1)
attn2q_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kv,
              const __grid_constant__ CUtensorMap tmap_o, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t sQ = s_base + Q2::kOffQ;
  const uint32_t sK = s_base + Q2::kOffK;
  const uint32_t sV = s_base + Q2::kOffV;
  const uint32_t sBar = s_base + Q2::kOffBar;
  uint8_t* misc = smem + Q2::kOffMisc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 16);
  // drains wait on their own control word, which nothing sets: after an abort
  // they still wait (bounded) for every copy and MMA in flight to complete
  volatile int* never_abort = reinterpret_cast<volatile int*>(misc + 20);
  volatile int* merge_flag = reinterpret_cast<volatile int*>(misc + 64);  // this CTA merges the unit
  auto bar = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };
  // PV(x, m) done: barrier 2 x + m % 2, phase m / 2
  auto pv_bar = [&](int x, uint32_t m) { return bar(kPV2A0 + 2 * x + static_cast<int>(m & 1u)); };
  auto pv_par = [&](uint32_t m) { return (m >> 1) & 1u; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const unsigned fullmask = 0xffffffffu;
  const WaitCtl ctl{abort_flag, p.err};
  const WaitCtl drain_ctl{never_abort, p.err};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *never_abort = 0;
    mbar_init(bar(kQ2Full), 1);
    mbar_init(bar(kQ2Empty), 1);
    for (int s = 0; s < Q2::kStages; ++s) {
      mbar_init(bar(kK2Full0 + s), 1);
      mbar_init(bar(kK2Empty0 + s), 1);
      mbar_init(bar(kV2Full0 + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(kS2Full0 + x), 1);
      mbar_init(bar(kP2Full0 + x), 4);
    }
    for (int i = 0; i < 4; ++i) mbar_init(bar(kPV2A0 + i), 1);
    mbar_init(bar(kDrain2), 1);
    mbar_init(bar(kDrainPV2), 1);
    mbar_init(bar(kMerge2A), kSoftmaxWarps);
    mbar_init(bar(kMerge2B), 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(kSl2Full0 + i), 4);
      mbar_init(bar(kSl2Free0 + i), 1);
    }
    mbar_init_fence();
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_kv);
    tma_prefetch_desc(&tmap_o);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  prefill_start(p, ctl);  // the plan (and whatever ran before it) is complete from here on
  grid_dep_launch();      // a dependent launch after this grid may take SMs as its CTAs leave

  const int n_items = p.hdr[kHdrItems];
  const int G = p.group;
  const int T = p.tokens_per_tile;
  const int cid = static_cast<int>(blockIdx.x);
  const int ncl = static_cast<int>(gridDim.x);

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ load warps
    // warp 0: both Q tiles of an item and the K tiles; warp 3: the V tiles. The
    // block table is read 32 tiles at a time across the lanes; lane 0 issues.
    const int kind = warp == 0 ? 0 : 1;
    const int full = kind ? kV2Full0 : kK2Full0;
    uint32_t n = 0, itl = 0;
    bool ok = true;
    const uint64_t pol_q = l2_policy_evict_last();
    const uint64_t pol_kv = l2_policy_evict_last();  // re-read by the sequence's other q tile pairs
    for (int kq = 0, idx = cid; idx < n_items && ok; idx = cta_item(++kq, cid, ncl), ++itl) {
      const Item it = decode_item(p.items[idx]);
      const int4 si = p.seq_info[it.b];
      const int q0 = si.x, ql = si.y, L = si.z, kv0 = si.w;
      if (kind == 0 && lane == 0) {
        ok = wait_one(bar(kQ2Empty), (itl & 1u) ^ 1u, ctl);
        if (ok) {
          const int ntq = (it.qt + 1) * T < ql ? 2 : 1;  // q tile B exists
          mbar_arrive_expect_tx(bar(kQ2Full), static_cast<uint32_t>(ntq * 2 * 128 * G * T));
          for (int x = 0; x < ntq; ++x)
            for (int c = 0; c < 2; ++c)
              tma_load_4d(sQ + x * Q2::kQBytes + c * (kBM * 128), &tmap_q, bar(kQ2Full), c * 64, 0, it.hk,
                          q0 + (it.qt + x) * T, pol_q);
        }
      }
      ok = __shfl_sync(fullmask, ok, 0);
      const int ntiles = it.kt1 - it.kt0;
      for (int t0 = 0; t0 < ntiles && ok; t0 += 32) {
        // lane l looks up the two pages of tile t0 + l
        int pg[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          pg[j] = -1;
          const int key = (it.kt0 + t0 + lane) * kBN2 + j * kPage;
          if (t0 + lane < ntiles && key < L) {
            if (p.paged) {
              const int page = p.block_table[static_cast<size_t>(it.b) * p.bt_stride + key / kPage];
              if (page >= 0 && page < p.num_pages)
                pg[j] = page;
              else
                atomicOr(p.err, kErrBadInput);
            } else {
              pg[j] = kv0 + key;
            }
          }
        }
        const int nb = min(32, ntiles - t0);
        for (int i = 0; i < nb; ++i, ++n) {
          int a[2];
          int nload = 0;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            a[j] = __shfl_sync(fullmask, pg[j], i);
            nload += a[j] >= 0;
          }
          if (lane == 0) {
            const uint32_t st = n % Q2::kStages;
            if (kind == 0)
              ok = wait_one(bar(kK2Empty0 + st), ((n / Q2::kStages) & 1u) ^ 1u, ctl);
            else if (n >= static_cast<uint32_t>(Q2::kStages))
              // a V stage is free once both PVs of the tile it held are done
              ok = wait_one(pv_bar(1, n - Q2::kStages), pv_par(n - Q2::kStages), ctl);
            if (ok) {
              mbar_arrive_expect_tx(bar(full + st), static_cast<uint32_t>(nload * 2 * kPage * 128));
              const uint32_t dst0 = (kind ? sV : sK) + st * Q2::kStage;
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                if (a[j] < 0) continue;
                for (int c = 0; c < 2; ++c) {
                  const uint32_t dst = dst0 + c * (kBN2 * 128) + j * (kPage * 128);
                  if (p.paged)
                    tma_load_4d(dst, &tmap_kv, bar(full + st), c * 64, 0, it.hk, 2 * a[j] + kind, pol_kv);
                  else
                    tma_load_4d(dst, &tmap_kv, bar(full + st), c * 64, it.hk, a[j], kind, pol_kv);
                }
              }
            }
          }
          ok = __shfl_sync(fullmask, ok, 0);
          if (!ok) break;  // n counts only the fills that were issued
        }
      }
    }
    // Drain: every copy this warp started has landed before exit.
    if (lane == 0) {
      for (uint32_t st = 0; st < static_cast<uint32_t>(Q2::kStages); ++st) {
        if (n <= st) continue;
        const uint32_t last = ((n - 1 - st) / Q2::kStages) * Q2::kStages + st;  // last fill of stage st
        wait_one(bar(full + st), (last / Q2::kStages) & 1u, drain_ctl);
      }
      if (kind == 0 && itl > 0) wait_one(bar(kQ2Full), (itl - 1) & 1u, drain_ctl);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK MMA thread
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN2, false, false);
      const SmemDesc dq = sw128_desc_split(sQ, 16, 1024);
      const SmemDesc dk = sw128_desc_split(sK, 16, 1024);
      uint32_t n = 0, itl = 0;
      bool ok = true;
      // failure-detection self-test: the first CTA's QK thread first waits for a
      // phase that nothing completes before the drain below, so the wait runs
      // out and every role of the CTA takes its abort path
      if (p.selftest_abort && blockIdx.x == 0 && n_items > 0) ok = wait_one(bar(kDrain2), 0, ctl);
      for (int kq = 0, idx = cid; idx < n_items && ok; idx = cta_item(++kq, cid, ncl), ++itl) {
        const Item it = decode_item(p.items[idx]);
        const bool has_b = (it.qt + 1) * T < p.seq_info[it.b].y;
        if (!(ok = wait_one(bar(kQ2Full), itl & 1u, ctl))) break;
        tc_fence_after();
        for (int kt = it.kt0; kt < it.kt1; ++kt, ++n) {
          const uint32_t ks = n % Q2::kStages;
          if (!(ok = wait_one(bar(kK2Full0 + ks), (n / Q2::kStages) & 1u, ctl))) break;
          const uint32_t k_lo = desc_lo_at(dk, ks * Q2::kStage);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            // S_X is free once PV(X, n - 1) has read P_X over it
            if (n > 0 && !(ok = wait_one(pv_bar(x, n - 1), pv_par(n - 1), ctl))) break;
            tc_fence_after();
            if (x == 0 || has_b) {
              const uint32_t q_lo = desc_lo_at(dq, x * Q2::kQBytes);
#pragma unroll
              for (int kk = 0; kk < kD2 / 16; ++kk) {
                const uint32_t b_lo = k_lo + (((kk >> 2) * (kBN2 * 128) + (kk & 3) * 32) >> 4);
                const uint32_t a_lo = q_lo + (((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
                umma_f16_ss(tmem + Q2::kColS + x * kBN2, a_lo, dq.hi, b_lo, dk.hi, idesc_qk, kk > 0 ? 1u : 0u);
              }
            }
            umma_commit(bar(kS2Full0 + x));  // (no MMA for an absent q tile B: the phase still completes)
          }
          if (!ok) break;
          umma_commit(bar(kK2Empty0 + ks));  // both QKs of the tile have read K
        }
        if (!ok) break;
        umma_commit(bar(kQ2Empty));  // the item's last QKs have read both Q tiles
      }
      // Drain: all UMMAs issued by this thread complete before TMEM is freed.
      umma_commit(bar(kDrain2));
      wait_one(bar(kDrain2), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ V tail + PV MMA thread
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, kD2, false, true);
    const SmemDesc dv = sw128_desc_split(sV, kBN2 * 128, 1024);  // V MN-major
    uint32_t n = 0;
    bool ok = true;
    for (int kq = 0, idx = cid; idx < n_items && ok; idx = cta_item(++kq, cid, ncl)) {
      const Item it = decode_item(p.items[idx]);
      const int4 si = p.seq_info[it.b];
      const int L = si.z;
      const bool has_b = (it.qt + 1) * T < si.y;
      for (int kt = it.kt0; kt < it.kt1; ++kt, ++n) {
        const uint32_t s = n % Q2::kStages;
        if (!(ok = wait_warp(bar(kV2Full0 + s), (n / Q2::kStages) & 1u, ctl))) break;
        const int live = L - kt * kBN2;
        if (live < kBN2) {
          // whole 128-byte rows past the sequence end (the swizzle does not matter)
          uint8_t* v0 = smem + Q2::kOffV + s * Q2::kStage;
          const int chunks = (kBN2 - live) * 8;  // 16-byte chunks per 64-column block
          for (int c = 0; c < 2; ++c) {
            uint4* blk = reinterpret_cast<uint4*>(v0 + c * (kBN2 * 128) + live * 128);
            for (int i = lane; i < chunks; i += 32) blk[i] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          const bool first = kt == it.kt0;
          const uint32_t v_lo = desc_lo_at(dv, s * Q2::kStage);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!(ok = wait_one(bar(kP2Full0 + x), n & 1u, ctl))) break;
            tc_fence_after();
            if (x == 0 || has_b) {
#pragma unroll
              for (int kk = 0; kk < kBN2 / 16; ++kk) {
                const uint32_t b_lo = v_lo + ((kk * (16 * 128)) >> 4);
                umma_f16_ts(tmem + Q2::kColO + x * kD2, tmem + Q2::kColS + x * kBN2 + kk * 8, b_lo, dv.hi,
                            idesc_pv, (first && kk == 0) ? 0u : 1u);
              }
            }
            umma_commit(pv_bar(x, n));  // P_X and (after B) the V stage are free
          }
        }
        ok = __shfl_sync(fullmask, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0) {
      umma_commit(bar(kDrainPV2));
      wait_one(bar(kDrainPV2), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax of q tile x
    const int x = (warp - 4) >> 2;       // 0: q tile A (qt), 1: q tile B (qt + 1)
    const int sw = (warp - 4) & 3;       // TMEM lane quarter
    const int r = sw * 32 + lane;        // packed query row of this thread
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    const uint32_t s_col = tmem + lane_base + Q2::kColS + x * kBN2;
    const uint32_t o_col = tmem + lane_base + Q2::kColO + x * kD2;
    const int t_local = r / G;
    const int g = r - t_local * G;
    const float c = p.scale_log2;
    uint32_t n = 0, n_split = 0;
    uint32_t n_slice = 0;  // output slices staged by this warpgroup
    bool ok = true;
    int4 iv_next = cid < n_items ? p.items[cid] : make_int4(0, 0, 0, 0);
    int4 si_next = cid < n_items ? p.seq_info[iv_next.x & kSeqMask] : make_int4(0, 0, 0, 0);
    for (int kq = 0, idx = cid; idx < n_items && ok; idx = cta_item(++kq, cid, ncl)) {
      const Item it = decode_item(iv_next);
      const int4 si = si_next;
      const int idx_next = cta_item(kq + 1, cid, ncl);
      const bool has_next = idx_next < n_items;
      if (has_next) iv_next = p.items[idx_next];
      const int q0 = si.x, ql = si.y, L = si.z;
      const int qtx = it.qt + x;
      const int tok = qtx * T + t_local;
      const bool valid = (t_local < T) && (tok < ql);
      int lim = 0;  // keys [0, lim) visible to this row
      if (valid) lim = p.causal ? min(L, L - ql + tok + 1) : L;
      const bool warp_live = __any_sync(fullmask, valid) != 0;
      float m_used = -INFINITY, l = 0.f;
      for (int kt = it.kt0; kt < it.kt1; ++kt, ++n) {
        const bool first = kt == it.kt0;
        if (!(ok = wait_warp(bar(kS2Full0 + x), n & 1u, ctl))) break;
        tc_fence_after();
        if (kt + 1 == it.kt1 && has_next) si_next = p.seq_info[iv_next.x & kSeqMask];
        if (warp_live) {
          const int nv = lim - kt * kBN2;  // visible keys of this row in the tile (any sign)
          const bool full_tile = nv >= kBN2;
          // P of the whole row (128 keys as 64 bf16 pairs), computed against the
          // running max first: a row sum of at most 2^8 bounds every p by 2^8,
          // exactly the case in which the running max is kept. Otherwise (and on
          // an item's first tile) the tile max decides and P is recomputed.
          uint32_t pk[64];
          auto exp_pass = [&](float m_ref) -> float {
            float sum = 0.f;
#pragma unroll
            for (int c2 = 0; c2 < 4; c2 += 2) {
              uint32_t sa[32], sb[32];
              tmem_ld32(s_col + c2 * 32, sa);
              tmem_ld32(s_col + (c2 + 1) * 32, sb);
              tmem_wait_ld();
              reg_fence(sa);
              reg_fence(sb);
              uint32_t(&pa)[16] = *reinterpret_cast<uint32_t(*)[16]>(&pk[c2 * 16]);
              uint32_t(&pb)[16] = *reinterpret_cast<uint32_t(*)[16]>(&pk[(c2 + 1) * 16]);
              if (full_tile) {
                sum += chunk_exp<false>(sa, c, m_ref, 32, pa) + chunk_exp<false>(sb, c, m_ref, 32, pb);
              } else {
                sum += chunk_exp<true>(sa, c, m_ref, nv - c2 * 32, pa) +
                       chunk_exp<true>(sb, c, m_ref, nv - (c2 + 1) * 32, pb);
              }
            }
            return sum;
          };
          // (warp-uniform: every lane runs the same tensor-memory loads. A row that
          // has seen no key yet has m_used = -inf: its visible keys give an
          // infinite sum, which takes the exact path; masked keys give p = 0.)
          const float kSumLimit = 256.0f;
          float lt = 0.f;
          bool exact = first;
          if (!first) {
            lt = exp_pass(m_used);
            exact = !(lt <= kSumLimit);  // also true for inf / NaN
          }
          if (__any_sync(fullmask, exact)) {
            // the tile max, two chunks per round trip to tensor memory
            float mx = -INFINITY;
#pragma unroll
            for (int c2 = 0; c2 < 4; c2 += 2) {
              uint32_t sa[32], sb[32];
              tmem_ld32(s_col + c2 * 32, sa);
              tmem_ld32(s_col + (c2 + 1) * 32, sb);
              tmem_wait_ld();
              reg_fence(sa);
              reg_fence(sb);
              if (full_tile) {
                mx = fmaxf(mx, fmaxf(chunk_max<false>(sa, 32), chunk_max<false>(sb, 32)));
              } else {
                mx = fmaxf(mx, fmaxf(chunk_max<true>(sa, nv - c2 * 32), chunk_max<true>(sb, nv - (c2 + 1) * 32)));
              }
            }
            const float mx_s = (mx == -INFINITY) ? -INFINITY : mx * c;
            const float m_new = fmaxf(m_used, mx_s);
            if (first) {
              m_used = m_new;  // O starts over on the item's first tile
            } else {
              const bool need = m_new > m_used + 8.0f;
              if (__any_sync(fullmask, need)) {
                // O_X holds the previous tiles; rescale it once their PV is done
                const uint32_t pm = n - 1;
                if (!(ok = wait_warp(pv_bar(x, pm), pv_par(pm), ctl))) break;
                tc_fence_after();
                const float alpha = need ? ex2(m_used - m_new) : 1.0f;
                if (need) {
                  l *= alpha;
                  m_used = m_new;
                }
#pragma unroll 1
                for (int j = 0; j < kD2 / 32; ++j) {
                  uint32_t o[32];
                  tmem_ld32(o_col + j * 32, o);
                  tmem_wait_ld();
                  reg_fence(o);
#pragma unroll
                  for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                  tmem_st32(o_col + j * 32, o);
                }
                tmem_wait_st();
              }
            }
            lt = exp_pass((m_used == -INFINITY) ? 0.f : m_used);
          }
          l += lt;
          // P over the first 64 columns of S_X (all of S has been read)
          tmem_st32(s_col, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          tmem_st32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kP2Full0 + x));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      {
        const uint32_t pm = n - 1;  // the item's last PV of this q tile
        if (!(ok = wait_warp(pv_bar(x, pm), pv_par(pm), ctl))) break;
      }
      tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      const bool tma_out = it.part < 0 && (qtx + 1) * T <= ql;
      if (tma_out) {
        // a full q tile of an unsplit item: four 32-column slices staged in
        // shared memory (two buffers, used in turn), each stored as the box
        // [32 channels, G heads, 1, T tokens]. The hand-offs are bounded mbarrier
        // waits (slice staged by all four warps -> the issuing thread stores it;
        // the store of the slice after it has been issued -> its buffer is free
        // again), so that a warp that gave up elsewhere cannot leave the others
        // waiting.
        const uint32_t sx = static_cast<uint32_t>((r >> 1) & 3);  // 64-byte swizzle of this row
#pragma unroll 1
        for (int pp = 0; pp < kD2 / 32 && ok; ++pp, ++n_slice) {
          const int col = pp * 32;
          const int sb = 2 * x + static_cast<int>(n_slice & 1u);  // slice buffer
          const uint32_t use = n_slice >> 1;                        // its use count
          const uint32_t stage = s_base + Q2::kOffO + static_cast<uint32_t>(sb * Q2::kOSlice);
          const uint32_t row_addr = stage + static_cast<uint32_t>(r * 64);
          // the buffer is free once the store of its previous use has read it
          if (!(ok = wait_warp(bar(kSl2Free0 + sb), (use & 1u) ^ 1u, ctl))) break;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t o[16];
            tmem_ld16(o_col + col + hf * 16, o);
            tmem_wait_ld();
            reg_fence(o);
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              __nv_bfloat162 hh =
                  __floats2bfloat162_rn(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
              w[e] = *reinterpret_cast<uint32_t*>(&hh);
            }
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
              st_shared_v4(row_addr + ((static_cast<uint32_t>(2 * hf + c2) ^ sx) << 4), w[4 * c2],
                           w[4 * c2 + 1], w[4 * c2 + 2], w[4 * c2 + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kSl2Full0 + sb));
          if (sw == 0) {
            if (lane == 0) {
              ok = wait_one(bar(kSl2Full0 + sb), use & 1u, ctl);
              if (ok) {
                tma_store_4d(&tmap_o, stage, col, 0, it.hk, q0 + qtx * T);
                bulk_commit_group();
                // the store before this one has read its buffer: free it
                if (n_slice > 0) {
                  bulk_wait_read_1();
                  mbar_arrive(bar(kSl2Free0 + 2 * x + static_cast<int>((n_slice - 1) & 1u)));
                }
              }
            }
            ok = __shfl_sync(fullmask, ok, 0);
          }
        }
        if (!ok) break;
      } else if (warp_live) {
        const int hq = it.hk * G + g;
#pragma unroll 1
        for (int j = 0; j < kD2 / 16; ++j) {
          const int col = j * 16;
          uint32_t o[16];
          tmem_ld16(o_col + col, o);
          tmem_wait_ld();
          reg_fence(o);
          if (!valid) continue;
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(o[i]) * inv;
          if (it.part < 0) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(q0 + tok) * p.n_heads_q + hq) * kD2 + col);
#pragma unroll
            for (int q4 = 0; q4 < 2; ++q4) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 hh = __floats2bfloat162_rn(v[q4 * 8 + 2 * e], v[q4 * 8 + 2 * e + 1]);
                w[e] = *reinterpret_cast<uint32_t*>(&hh);
              }
              dst[q4] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            // a split item (one q tile: x = 0): the normalised partial O row
            float4* dst = reinterpret_cast<float4*>(p.part_o + static_cast<size_t>(it.part + r) * kD2 + col);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              dst[q4] = make_float4(v[q4 * 4], v[q4 * 4 + 1], v[q4 * 4 + 2], v[q4 * 4 + 3]);
          }
        }
        if (valid && it.part >= 0) p.part_ml[it.part + r] = make_float2(l > 0.f ? m_used : -INFINITY, l);
      }
      tc_fence_before();
      if (it.part >= 0 &&
          !(ok = split_done<kD2>(p, it, si, bar(kMerge2A), bar(kMerge2B), merge_flag, n_split, warp, ctl)))
        break;
    }
    // the output stores of this warpgroup complete before the CTA exits
    if (sw == 0 && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  prefill_end(p);
}

}  // namespace

cudaError_t attention2q_set_attributes() {
  return cudaFuncSetAttribute(attn2q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Q2::kSmem);
}

cudaError_t launch_attention_2q(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tkv,
                                const CUtensorMap& to, int grid, cudaStream_t s, bool dependent) {
  return launch_kernel(attn2q_kernel, grid, kThreads2, Q2::kSmem, s, dependent, tq, tkv, to, p);
}

}  // namespace pattn
