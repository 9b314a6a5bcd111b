// attn.cu -- fused paged-KV attention for sm_103a (tcgen05 + TMA): the prefill
// kernel, for work units of more than 16 packed query rows.
//
// One persistent CTA per SM walks the planned work list (longest first,
// round robin over CTAs). A work item is (sequence, kv head, q tile, KV tile
// range). Warp roles:
//
//   * warps 0 and 3 TMA-load the GQA-packed Q tile (the G query heads of one KV
//     head for T = 128 / G tokens, as 128 rows of 128-byte-swizzled shared
//     memory: the GQA-packed Q tensor map of the trtllm-gen paged decode
//     manifest, dims [D, group, kv head, token]) and, per KV tile of BN keys,
//     the K (warp 0) and V (warp 3) rows page by page through one tensor map
//     over the whole pool, [D, 64 rows, Hkv, 2 x pages] (the manifest's K and V
//     maps), each page read once per KV head for all G query heads;
//   * warp 1 issues S = Q K^T (tcgen05.mma kind::f16, M = 128, N = BN, K = D)
//     from one thread, both operands from shared memory;
//   * warp 2 zeroes V rows past the sequence end (so that NaN or garbage there
//     cannot reach O through 0 * NaN) and issues O += P V (M = 128, N = D,
//     K = BN) with P from TMEM and V read MN-major from shared memory. QK and
//     PV come from different threads so that each stream's waits overlap the
//     other's MMAs; commits signal mbarriers (the SM100MHA2Q "UMMA0" / "UMMA1"
//     accumulators of the FlashAttention-4 doc);
//   * warps 4-11 are two softmax warpgroups over the same 128 query rows, one
//     row per thread in each, splitting the keys of every tile between them
//     (D = 256: sharing one O accumulator in TMEM). Each reads its half of the S row,
//     computes P = 2^(S c - m) against the running max m (log2 units, the scale
//     folded into log2 e, as the manifest's pack scalar does) and writes P as
//     bf16 pairs into TMEM, where the PV MMA reads its A operand. The two warps
//     of a row pair then add up their halves of the row sum: a sum of at most
//     2^8 bounds every p by 2^8, which is exactly when the running max is kept.
//     Otherwise (and on an item's first tile) they exchange the tile max, O is
//     rescaled in TMEM if the max grew by more than 2^8 (exact: O and l share
//     the stale max), and P is recomputed.
//
// D = 128 keeps one O per warpgroup instead (each over its own key half, with
// its own running max, merged once per item), so that the warpgroups need not
// agree on anything per tile; each skips the tile max while the sum of its
// probabilities against its running max stays at most 2^8.
//
// TMEM (512 columns): D = 128: O0 | O1 | S0 | S1, P written over the S columns
// each warp has just read, so that QK of tile n waits only for the PV of tile
// n - 2. D = 256: O | S0 | S1 | P0 | P1.
//
// Quantised instances (head_dim 128): kF8 takes e4m3 Q and K codes for S (four
// kind::f8f6f4 MMAs of K = 32) and scales each warpgroup's scores by the Q row
// and K block scales. kF8V also codes P and V: the softmax computes the tile
// max only when needed (as for bf16 P, with its own limits), writes e4m3 of
// p * 2^2 (at most 2^8, inside the e4m3 range) into TMEM over the S columns it has just
// read (four codes per column), and O += P V runs as kind::f8f6f4 MMAs with P
// from TMEM and V from shared memory as transposed e4m3 tiles (K-major); the
// per-channel V scale is applied in the epilogue.
//
// At the end of an item the softmax warps divide by l and store bf16 rows (at
// head_dim 128, a full q tile of an unsplit item as 32-column slices staged in
// shared memory and written by a tensor store), or (split items) write the
// normalised partial O and (m, l), count the split in its unit, and the CTA
// that finishes a unit's last split merges it.
#include <cuda_fp8.h>

#include "kernels.cuh"
#include "merge.cuh"
#include "prefill.cuh"
#include "ptx.cuh"

namespace pattn {
namespace {

template <int D, int BN, bool kF8 = false, bool kF8V = false, bool kPair = false>
struct Cfg {
  // kF8: Q and K as e4m3 codes (one byte), S = Q K^T with kind::f8f6f4 MMAs; V
  // stays bf16 unless kF8V (P and V e4m3, P in TMEM).
  // kPair: a CTA pair shares each tile's MMAs (cta_group::2): a CTA holds its
  // own q tile, half of the K rows (one page) and half of the V columns.
  static_assert(!kF8V || (kF8 && D == 128 && BN == 128), "fp8 P.V: head_dim 128, 128-key tiles");
  static_assert(!kPair || (D == 256 && BN == 128 && !kF8), "CTA pairs: head_dim 256, 128-key tiles, bf16");
  static constexpr int kQKElem = kF8 ? 1 : 2;          // bytes per Q / K element
  static constexpr int kQBytes = kBM * D * kQKElem;
  static constexpr int kKRows = kPair ? BN / 2 : BN;   // K rows of a tile held by this CTA
  static constexpr int kKStage = kKRows * D * kQKElem;
  static constexpr int kVCols = kPair ? D / 2 : D;     // V columns of a tile held by this CTA
  static constexpr int kVStage = BN * kVCols * (kF8V ? 1 : 2);
  static constexpr int kQKBlocks = D * kQKElem / 128;  // 128-byte swizzle columns of a Q / K row
  static constexpr int kQKBlockElems = 128 / kQKElem;
  static constexpr int kQKSteps = D * kQKElem / 32;    // MMAs of one QK (32 bytes of K each)
  static constexpr bool kSplitO = D == 128;          // one O per softmax warpgroup
  static constexpr bool kAliasP = D == 128 || kPair;  // P over its S buffer
  static constexpr int kSBufs = 2;
  static constexpr int kPBufs = kAliasP ? kSBufs : 2;
  static constexpr int kPVBars = kAliasP ? kSBufs : 2;  // pv_done barriers, by tile index
  static constexpr int kQBufs = D == 128 ? 2 : 1;    // D = 128: the next item's Q lands early
  static constexpr int kKStages = kF8V ? 3 : 2;       // e4m3 tiles are half as large
  static constexpr int kVStages = kF8V ? 3 : 2;
  // shared memory
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBufs * kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKStage;
  // D = 128: each warpgroup stages a 32-column slice of its bf16 output rows
  // (64-byte rows, 64-byte swizzle) for the tensor store
  static constexpr int kOStage = kSplitO ? 2 * kBM * 64 : 0;
  static constexpr int kOffO = kOffV + kVStages * kVStage;
  static constexpr int kOffX = kOffO + kOStage;  // row sum / max / l exchange
  static constexpr int kXBytes = (2 * 2 + 2 * 2 + 2) * kBM * 4;
  static constexpr int kOffBar = kOffX + kXBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kOffMisc = kOffBar + kBarBytes;
  static constexpr int kSmem = kOffMisc + 128 + 1024;  // + alignment slack
  // tensor memory
  static constexpr int kColO = 0;
  static constexpr int kColS = kSplitO ? 2 * D : D;
  static constexpr int kPCols = BN / 2;               // P as bf16 pairs: BN keys in BN/2 columns
  static constexpr int kColP = kColS + kSBufs * BN;   // separate P buffers (not aliased)
  // TMEM column of P buffer b for keys [16 kk, 16 kk + 16): over its own S
  // buffer (each warpgroup's half at the start of the half it read), or in a P
  // buffer.
  // kF8V: e4m3 P, keys [32 kk, 32 kk + 32) in 8 columns over S the same way.
  __device__ static constexpr int p_col(int b, int kk) {
    return kF8V ? kColS + b * BN + (kk / (BN / 64)) * (BN / 2) + (kk % (BN / 64)) * 8
           : kAliasP ? kColS + b * BN + (kk / (BN / 32)) * (BN / 2) + (kk % (BN / 32)) * 8
                     : kColP + b * kPCols + kk * 8;
  }
  static constexpr int kDBlocks = kVCols / 64;        // 128-byte swizzle columns of this CTA's V rows
  static constexpr int kPagesPerTile = BN / kPage;
  static_assert(kColS + kSBufs * BN + ((kAliasP || kF8V) ? 0 : kPBufs * kPCols) <= kTmemCols, "TMEM budget");
  static_assert(kSBufs <= 3 && kPBufs <= 3 && kPVBars <= 3 && kQBufs <= 2, "barrier slots");
  static_assert(kKStages <= 3 && kVStages <= 3, "ring barrier slots");
  // bf16 V stages are released through the pv_done barrier of their tile, e4m3
  // ones through their own empty barriers
  static_assert(kF8V || kVStages <= kPVBars, "V stage release");
  static_assert((kSplitO ? 2 * D : D) <= kColS, "O columns");
  static_assert(BN % kPage == 0 && BN % 32 == 0, "tile");
  static_assert(kSmem <= 232448, "shared memory budget");
};

// mbarrier slots
enum Bar {
  kQFull0 = 0, kQFull1, kQEmpty0, kQEmpty1, kKFull0, kKFull1, kKFull2, kKEmpty0, kKEmpty1, kKEmpty2,
  kVFull0, kVFull1, kVFull2, kVEmpty0, kVEmpty1, kVEmpty2, kSFull0, kSFull1, kSFull2, kSFree0, kSFree1, kSFree2, kPFull0, kPFull1, kPFull2, kPVDone0,
  kPVDone1, kPVDone2, kDrain, kDrainPV, kPairA0, kPairA1, kPairA2, kPairA3, kPairB0, kPairB1,
  kPairB2, kPairB3, kXSum,
  // CTA pairs, in the rank-0 CTA: the peer's Q, K stage and V stage are ready
  kPeerQ, kPeerK0, kPeerK1, kPeerK2, kPeerV0, kPeerV1, kPeerV2,
  // split items: every softmax warp's partials written; the unit counter read
  kMergeA, kMergeB,
  // head_dim 128 output slices: warpgroup h's rows staged (4 warps); its buffer read by the store
  kOSlFull0, kOSlFull1, kOSlFree0, kOSlFree1, kNumBars
};
static_assert(kNumBars * 8 <= 512, "mbarrier area");
constexpr int kAttnThreads = 384;  // load K, MMA, V tail, load V; 2 softmax warpgroups

// One row's probabilities for KH keys: p_i = 2^(S_i c - m_ref) as bf16 pairs in
// pk, returning the fp32 sum of the p_i. With kMasked only the first nv keys
// count (the others give 0 whatever their score); full tiles take the unmasked
// body, so they carry no per-key compare. Scale and sum use packed fp32x2 ops.
template <int KH, bool kMasked>
__device__ __forceinline__ float exp_row(const uint32_t (&sr)[KH / 32][32], float c, float m_ref,
                                         int nv, uint32_t (&pk)[KH / 2]) {
  const float2 c2 = make_float2(c, c);
  const float2 nm2 = make_float2(-m_ref, -m_ref);
  float2 acc[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) acc[u] = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < KH / 32; ++j) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 x =
          __ffma2_rn(make_float2(__uint_as_float(sr[j][i]), __uint_as_float(sr[j][i + 1])), c2, nm2);
      float p0 = ex2(x.x);
      float p1 = ex2(x.y);
      if constexpr (kMasked) {
        p0 = j * 32 + i < nv ? p0 : 0.f;
        p1 = j * 32 + i + 1 < nv ? p1 : 0.f;
      }
      acc[(i >> 1) & 3] = __fadd2_rn(acc[(i >> 1) & 3], make_float2(p0, p1));
      __nv_bfloat162 hh = __floats2bfloat162_rn(p0, p1);
      pk[(j * 32 + i) >> 1] = *reinterpret_cast<uint32_t*>(&hh);
    }
  }
  const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  return a.x + a.y;
}

// The same for the fp8 P.V instance: p_i = 2^(S_i c - m_ref) with m_ref the
// running max minus 2 (p scaled by 2^2), as e4m3 codes, four per word in key
// order, returning the fp32 sum of the unrounded p_i.
template <int KH, bool kMasked>
__device__ __forceinline__ float exp_row_f8(const uint32_t (&sr)[KH / 32][32], float c, float m_ref,
                                            int nv, uint32_t (&pk)[KH / 4]) {
  const float2 c2 = make_float2(c, c);
  const float2 nm2 = make_float2(-m_ref, -m_ref);
  float2 acc[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) acc[u] = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < KH / 32; ++j) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      uint32_t w = 0;
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const int k = i + 2 * hv;
        const float s0 = __uint_as_float(sr[j][k]), s1 = __uint_as_float(sr[j][k + 1]);
        const float2 x = __ffma2_rn(make_float2(s0, s1), c2, nm2);
        float p0 = ex2(x.x);
        float p1 = ex2(x.y);
        if constexpr (kMasked) {
          p0 = j * 32 + k < nv ? p0 : 0.f;
          p1 = j * 32 + k + 1 < nv ? p1 : 0.f;
        }
        acc[(k >> 1) & 3] = __fadd2_rn(acc[(k >> 1) & 3], make_float2(p0, p1));
        const uint32_t pair = static_cast<uint32_t>(
            __nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE, __NV_E4M3));
        w |= pair << (16 * hv);
      }
      pk[(j * 32 + i) >> 2] = w;
    }
  }
  const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  return a.x + a.y;
}

// Max of the first nv of a row's KH scores (all of them when !kMasked).
template <int KH, bool kMasked>
__device__ __forceinline__ float max_row(const uint32_t (&sr)[KH / 32][32], int nv) {
  float acc[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) acc[u] = -INFINITY;
#pragma unroll
  for (int j = 0; j < KH / 32; ++j)
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (!kMasked || j * 32 + i < nv) acc[i & 7] = fmaxf(acc[i & 7], __uint_as_float(sr[j][i]));
  return fmaxf(fmaxf(fmaxf(acc[0], acc[1]), fmaxf(acc[2], acc[3])),
               fmaxf(fmaxf(acc[4], acc[5]), fmaxf(acc[6], acc[7])));
}

template <int D, int BN, bool kF8, bool kF8V, bool kPair>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kv,
            const __grid_constant__ CUtensorMap tmap_k8, const __grid_constant__ CUtensorMap tmap_v8,
            const __grid_constant__ CUtensorMap tmap_o, const AttnParams p) {
  using C = Cfg<D, BN, kF8, kF8V, kPair>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t sQ = s_base + C::kOffQ;
  const uint32_t sK = s_base + C::kOffK;
  const uint32_t sV = s_base + C::kOffV;
  const uint32_t sBar = s_base + C::kOffBar;
  uint8_t* misc = smem + C::kOffMisc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 16);
  // drains wait on their own control word, which nothing sets: after an abort
  // they still wait (bounded) for every copy and MMA in flight to complete
  volatile int* never_abort = reinterpret_cast<volatile int*>(misc + 20);
  volatile int* merge_flag = reinterpret_cast<volatile int*>(misc + 64);  // this CTA merges the unit
  // CTA pairs: 16-byte source and destination of the peer's signalling copies
  const uint32_t sig_src = smem_addr(misc + 32), sig_dst = smem_addr(misc + 48);
  auto bar = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };
  // pv_done of tile m: barrier m % kPVBars, phase m / kPVBars
  auto pv_bar = [&](uint32_t m) { return bar(kPVDone0 + static_cast<int>(m % C::kPVBars)); };
  auto pv_par = [&](uint32_t m) { return (m / C::kPVBars) & 1u; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtl ctl{abort_flag, p.err};
  const WaitCtl drain_ctl{never_abort, p.err};
  // CTA pairs walk the item list together (pair c = CTAs 2c, 2c + 1); the
  // rank-0 CTA issues the MMAs of both
  const uint32_t rank = kPair ? cluster_rank() : 0u;
  const int cid = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ncl = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *never_abort = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kQFull0 + b), 1);
      mbar_init(bar(kQEmpty0 + b), 1);  // the item's last QK MMA releases the buffer
    }
    for (int b = 0; b < 3; ++b) {
      mbar_init(bar(kKFull0 + b), 1);
      mbar_init(bar(kKEmpty0 + b), 1);
      mbar_init(bar(kVFull0 + b), 1);
      mbar_init(bar(kVEmpty0 + b), 1);
      mbar_init(bar(kSFull0 + b), 1);
      mbar_init(bar(kSFree0 + b), kSoftmaxWarps);
      // both key halves of P written; in the rank-0 CTA of a pair also the
      // PV thread's arrival that posts the peer's 16-byte signal
      mbar_init(bar(kPFull0 + b), (kPair && rank == 0) ? kSoftmaxWarps + 1 : kSoftmaxWarps);
      mbar_init(bar(kPeerK0 + b), 1);
      mbar_init(bar(kPeerV0 + b), 1);
      mbar_init(bar(kPVDone0 + b), 1);             // also frees that tile's V stage
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(bar(kPairA0 + b), 2);  // the two warps of a row quarter: row sums
      mbar_init(bar(kPairB0 + b), 2);  // and, when needed, row maxes
    }
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kDrainPV), 1);
    mbar_init(bar(kXSum), kSoftmaxWarps);
    mbar_init(bar(kPeerQ), 1);
    mbar_init(bar(kMergeA), kSoftmaxWarps);
    mbar_init(bar(kMergeB), 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(kOSlFull0 + h), 4);
      mbar_init(bar(kOSlFree0 + h), 1);
    }
    mbar_init_fence();
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_kv);
    if constexpr (kF8) tma_prefetch_desc(&tmap_k8);
    if constexpr (kF8V) tma_prefetch_desc(&tmap_v8);
    if constexpr (C::kSplitO) tma_prefetch_desc(&tmap_o);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  prefill_start(p, ctl);  // the plan (and whatever ran before it) is complete from here on
  grid_dep_launch();      // a dependent launch after this grid may take SMs as its CTAs leave

  const int n_items = p.hdr[kHdrItems];
  const int G = p.group;
  const int T = p.tokens_per_tile;

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ load warps
    // warp 0 loads Q and the K tiles, warp 3 the V tiles, so that a K load never
    // queues behind the release of a V stage. Each warp reads the block table
    // 32 tiles at a time across its lanes; lane 0 issues the copies.
    const int kind = warp == 0 ? 0 : 1;
    const uint32_t stages = kind ? C::kVStages : C::kKStages;
    const int full = kind ? kVFull0 : kKFull0;
    const unsigned fullmask = 0xffffffffu;
    uint32_t n = 0, itl = 0;
    bool ok = true;
    const uint64_t pol_q = l2_policy_evict_last();
    for (int kq = 0, idx = cid; idx < n_items && ok;
         idx = cta_item(++kq, cid, ncl), ++itl) {
      const Item it = decode_item(p.items[idx]);
      const int4 si = p.seq_info[it.b];
      const int q0 = si.x, L = si.z, kv0 = si.w;
      const bool decode_like = si.y <= T;
      const uint64_t pol_kv = decode_like ? l2_policy_evict_first() : l2_policy_evict_last();
      if (kind == 0 && lane == 0) {
        const uint32_t qb = itl % C::kQBufs, qu = itl / C::kQBufs;
        ok = wait_one(bar(kQEmpty0 + qb), (qu & 1u) ^ 1u, ctl);
        if (ok) {
          mbar_arrive_expect_tx(bar(kQFull0 + qb), static_cast<uint32_t>(C::kQKBlocks * 128 * G * T));
          for (int c = 0; c < C::kQKBlocks; ++c)
            tma_load_4d(sQ + qb * C::kQBytes + c * (kBM * 128), &tmap_q, bar(kQFull0 + qb),
                        c * C::kQKBlockElems, 0, it.hk, q0 + (it.qt + static_cast<int>(rank)) * T, pol_q);
        }
      }
      ok = __shfl_sync(fullmask, ok, 0);
      const int ntiles = it.kt1 - it.kt0;
      for (int t0 = 0; t0 < ntiles && ok; t0 += 32) {
        // lane l looks up the pages of tile t0 + l
        int pg[C::kPagesPerTile];
#pragma unroll
        for (int j = 0; j < C::kPagesPerTile; ++j) {
          pg[j] = -1;
          const int key = (it.kt0 + t0 + lane) * BN + j * kPage;
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
          int a[C::kPagesPerTile];
          int nload = 0;
#pragma unroll
          for (int j = 0; j < C::kPagesPerTile; ++j) {
            a[j] = __shfl_sync(fullmask, pg[j], i);
            nload += a[j] >= 0;
          }
          if (lane == 0) {
            const uint32_t st = n % stages;
            if (kind == 0) {
              ok = wait_one(bar(kKEmpty0 + st), ((n / stages) & 1u) ^ 1u, ctl);
            } else if (kF8V) {
              ok = wait_one(bar(kVEmpty0 + st), ((n / stages) & 1u) ^ 1u, ctl);
            } else if (n >= stages) {
              // a V stage is free once the PV of the tile it held is done
              ok = wait_one(pv_bar(n - stages), pv_par(n - stages), ctl);
            }
            if (ok && kPair && kind == 0) {
              // this CTA's page of the tile: rank r holds keys [64 r, 64 r + 64)
              const int pgk = rank ? a[C::kPagesPerTile - 1] : a[0];
              mbar_arrive_expect_tx(bar(full + st), pgk >= 0 ? static_cast<uint32_t>((D / 64) * kPage * 128) : 0u);
              if (pgk >= 0) {
                for (int c = 0; c < D / 64; ++c) {
                  const uint32_t dst = sK + st * C::kKStage + c * (kPage * 128);
                  if (p.paged)
                    tma_load_4d(dst, &tmap_kv, bar(full + st), c * 64, 0, it.hk, 2 * pgk, pol_kv);
                  else
                    tma_load_4d(dst, &tmap_kv, bar(full + st), c * 64, it.hk, pgk, 0, pol_kv);
                }
              }
            } else if (ok && kPair) {
              // this CTA's half of the V columns, both pages
              mbar_arrive_expect_tx(bar(full + st), static_cast<uint32_t>(nload * C::kDBlocks * kPage * 128));
#pragma unroll
              for (int j = 0; j < C::kPagesPerTile; ++j) {
                if (a[j] < 0) continue;
                for (int c = 0; c < C::kDBlocks; ++c) {
                  const int gc = static_cast<int>(rank) * C::kDBlocks + c;
                  const uint32_t dst = sV + st * C::kVStage + c * (BN * 128) + j * (kPage * 128);
                  if (p.paged)
                    tma_load_4d(dst, &tmap_kv, bar(full + st), gc * 64, 0, it.hk, 2 * a[j] + 1, pol_kv);
                  else
                    tma_load_4d(dst, &tmap_kv, bar(full + st), gc * 64, it.hk, a[j], 1, pol_kv);
                }
              }
            } else if (ok && kF8V && kind == 1) {
              // transposed e4m3 V: the whole 128-key tile of this head in one box
              // (zero codes past the sequence end)
              mbar_arrive_expect_tx(bar(full + st), static_cast<uint32_t>(C::kVStage));
              tma_load_4d(sV + st * C::kVStage, &tmap_v8, bar(full + st), 0, 0, it.hk,
                          it.b * (p.nb_max / 2) + it.kt0 + t0 + i, pol_kv);
            } else if (ok) {
              const int blocks = (kF8 && kind == 0) ? C::kQKBlocks : C::kDBlocks;
              mbar_arrive_expect_tx(bar(full + st), static_cast<uint32_t>(nload * blocks * kPage * 128));
              const uint32_t dst0 = kind ? sV + st * C::kVStage : sK + st * C::kKStage;
#pragma unroll
              for (int j = 0; j < C::kPagesPerTile; ++j) {
                if (a[j] < 0) continue;
                if (kF8 && kind == 0) {
                  // e4m3 K: 64-key block (tile * pages per tile + j) of the sequence
                  const int kblk = it.b * p.nb_max + (it.kt0 + t0 + i) * C::kPagesPerTile + j;
                  tma_load_4d(dst0 + j * (kPage * 128), &tmap_k8, bar(full + st), 0, 0, it.hk, kblk, pol_kv);
                  continue;
                }
                for (int c = 0; c < C::kDBlocks; ++c) {
                  const uint32_t dst = dst0 + c * (BN * 128) + j * (kPage * 128);
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
    // Drain: every copy this warp started must have landed before exit.
    if (lane == 0) {
      for (uint32_t st = 0; st < stages; ++st) {
        if (n <= st) continue;
        const uint32_t last = ((n - 1 - st) / stages) * stages + st;  // last fill on stage st
        wait_one(bar(full + st), (last / stages) & 1u, drain_ctl);
      }
      if (kind == 0) {
        for (uint32_t b = 0; b < static_cast<uint32_t>(C::kQBufs); ++b) {
          if (itl <= b) continue;
          const uint32_t last = ((itl - 1 - b) / C::kQBufs) * C::kQBufs + b;  // last Q fill of buffer b
          wait_one(bar(kQFull0 + b), (last / C::kQBufs) & 1u, drain_ctl);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK MMA warp
    // S = Q K^T for every tile, issued by one thread. The PV MMAs come from warp 2:
    // the two streams touch disjoint TMEM (S / P, O) and feed the tensor pipe
    // independently, so that neither one's waits leave the pipe idle.
    if (kPair && rank != 0 && lane == 0) {
      // the peer of a pair: forward "Q / K stage landed here" to the rank-0 CTA,
      // whose thread issues the MMAs of both
      uint32_t n = 0, itl = 0;
      bool ok = true;
      for (int kq = 0, idx = cid; idx < n_items && ok; idx = cta_item(++kq, cid, ncl), ++itl) {
        const Item it = decode_item(p.items[idx]);
        if (!(ok = wait_one(bar(kQFull0), itl & 1u, ctl))) break;
        signal_remote_tx(sig_dst, sig_src, bar(kPeerQ), 0);
        for (int kt = it.kt0; kt < it.kt1; ++kt, ++n) {
          const uint32_t ks = n % C::kKStages;
          if (!(ok = wait_one(bar(kKFull0 + ks), (n / C::kKStages) & 1u, ctl))) break;
          signal_remote_tx(sig_dst, sig_src, bar(kPeerK0 + static_cast<int>(ks)), 0);
        }
      }
    } else if (lane == 0) {
      constexpr uint32_t idesc_qk = kF8 ? idesc_e4m3_f32(kBM, BN)
                                        : idesc_bf16_f32(kPair ? 2 * kBM : kBM, BN, false, false);
      // operand descriptors built once; each MMA adds a compile-time offset
      const SmemDesc dq = sw128_desc_split(sQ, 16, 1024);
      const SmemDesc dk = sw128_desc_split(sK, 16, 1024);
      uint32_t n = 0, itl = 0;
      bool ok = true;
      // failure-detection self-test (one-CTA kernels): the first CTA's QK thread
      // first waits for a phase that nothing completes before the drain below,
      // so the wait runs out and every role of the CTA takes its abort path
      if (!kPair && p.selftest_abort && blockIdx.x == 0 && n_items > 0) ok = wait_one(bar(kDrain), 0, ctl);
      int4 iv_next = cid < n_items ? p.items[cid] : make_int4(0, 0, 0, 0);
      for (int kq = 0, idx = cid; idx < n_items && ok;
         idx = cta_item(++kq, cid, ncl), ++itl) {
        const Item it = decode_item(iv_next);
        if (cta_item(kq + 1, cid, ncl) < n_items)
          iv_next = p.items[cta_item(kq + 1, cid, ncl)];
        const uint32_t qb = itl % C::kQBufs, qu = itl / C::kQBufs;
        if (!(ok = wait_one(bar(kQFull0 + qb), qu & 1u, ctl))) break;
        if (kPair) {
          mbar_arrive_expect_tx(bar(kPeerQ), 16);  // the peer's Q signal
          if (!(ok = wait_one_cl(bar(kPeerQ), itl & 1u, ctl))) break;
        }
        tc_fence_after();
        const uint32_t q_lo = desc_lo_at(dq, qb * C::kQBytes);
        for (int kt = it.kt0; kt < it.kt1; ++kt, ++n) {
          const uint32_t s = n % C::kSBufs;
          const uint32_t ks = n % C::kKStages;
          // S buffer s is free once the softmax has read it, or (P written over
          // it) once the PV of tile n - kSBufs has consumed that P
          const uint32_t free_bar = C::kAliasP ? pv_bar(n) : bar(kSFree0 + static_cast<int>(s));
          const uint32_t free_par = ((n / C::kSBufs) & 1u) ^ 1u;
          if (!(ok = wait_two(bar(kKFull0 + ks), (n / C::kKStages) & 1u, free_bar, free_par, ctl))) break;
          if (kPair) {
            mbar_arrive_expect_tx(bar(kPeerK0 + static_cast<int>(ks)), 16);  // the peer's K signal
            if (!(ok = wait_one_cl(bar(kPeerK0 + static_cast<int>(ks)), (n / C::kKStages) & 1u, ctl))) break;
          }
          tc_fence_after();
          const uint32_t k_lo = desc_lo_at(dk, ks * C::kKStage);
          // 32 bytes of K per MMA: 16 bf16 or 32 e4m3 elements
#pragma unroll
          for (int kk = 0; kk < C::kQKSteps; ++kk) {
            const uint32_t b_lo = k_lo + (((kk >> 2) * (C::kKRows * 128) + (kk & 3) * 32) >> 4);
            const uint32_t a_lo = q_lo + (((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
            if constexpr (kF8)
              umma_f8_ss(tmem + C::kColS + s * BN, a_lo, dq.hi, b_lo, dk.hi, idesc_qk, kk > 0 ? 1u : 0u);
            else if constexpr (kPair)
              umma_f16_ss_pair(tmem + C::kColS + s * BN, a_lo, dq.hi, b_lo, dk.hi, idesc_qk, kk > 0 ? 1u : 0u);
            else
              umma_f16_ss(tmem + C::kColS + s * BN, a_lo, dq.hi, b_lo, dk.hi, idesc_qk, kk > 0 ? 1u : 0u);
          }
          if constexpr (kPair) {
            umma_commit_pair(bar(kKEmpty0 + ks));
            umma_commit_pair(bar(kSFull0 + s));
            if (kt + 1 == it.kt1) umma_commit_pair(bar(kQEmpty0 + qb));
          } else {
            umma_commit(bar(kKEmpty0 + ks));
            umma_commit(bar(kSFull0 + s));
            if (kt + 1 == it.kt1) umma_commit(bar(kQEmpty0 + qb));  // item's last QK
          }
        }
      }
      // Drain: all UMMAs issued by this thread complete before TMEM is freed.
      if constexpr (kPair) umma_commit_pair(bar(kDrain));
      else umma_commit(bar(kDrain));
      wait_one(bar(kDrain), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ V tail + PV MMA warp
    // Zeroes the V rows past the sequence end in a stage (whole 128-byte rows, so
    // the swizzle does not matter), then one thread issues O += P V for the tile.
    constexpr uint32_t idesc_pv =
        kF8V ? idesc_e4m3_f32(kBM, D) : idesc_bf16_f32(kPair ? 2 * kBM : kBM, D, false, true);
    // bf16 V: MN-major; e4m3 V: K-major transposed tiles, like the P buffers
    const SmemDesc dv = kF8V ? sw128_desc_split(sV, 16, 1024) : sw128_desc_split(sV, BN * 128, 1024);
    const unsigned fullmask = 0xffffffffu;
    uint32_t n = 0;
    bool ok = true;
    int4 iv_next = cid < n_items ? p.items[cid] : make_int4(0, 0, 0, 0);
    int L_next = cid < n_items ? p.seq_info[iv_next.x & kSeqMask].z : 0;
    for (int kq = 0, idx = cid; idx < n_items && ok; idx = cta_item(++kq, cid, ncl)) {
      const Item it = decode_item(iv_next);
      const int L = L_next;
      if (cta_item(kq + 1, cid, ncl) < n_items) {
        iv_next = p.items[cta_item(kq + 1, cid, ncl)];
        L_next = p.seq_info[iv_next.x & kSeqMask].z;
      }
      for (int kt = it.kt0; kt < it.kt1; ++kt, ++n) {
        const uint32_t s = n % C::kVStages;
        if (!(ok = wait_warp(bar(kVFull0 + s), (n / C::kVStages) & 1u, ctl))) break;
        const int live = L - kt * BN;
        if (!kF8V && live < BN) {
          uint8_t* v0 = smem + C::kOffV + s * C::kVStage;
          const int dead = BN - live;
          const int chunks = dead * 8;  // 16-byte chunks per block
          for (int c = 0; c < C::kDBlocks; ++c) {
            uint4* blk = reinterpret_cast<uint4*>(v0 + c * (BN * 128) + live * 128);
            for (int i = lane; i < chunks; i += 32) blk[i] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (kPair && rank != 0) {
          // the peer of a pair: its V half (tail zeroed), then its P, are ready for
          // the rank-0 CTA's PV. One remote arrive per tile: its softmax warps
          // arrive here, on their own CTA's barrier.
          if (lane == 0) {
            signal_remote_tx(sig_dst, sig_src, bar(kPeerV0 + static_cast<int>(s)), 0);
            const uint32_t pb = n % C::kPBufs, pu = n / C::kPBufs;
            ok = wait_one(bar(kPFull0 + pb), pu & 1u, ctl);
            tc_fence_after();
            tc_fence_before();
            if (ok) signal_remote_tx(sig_dst, sig_src, bar(kPFull0 + pb), 0);
          }
          ok = __shfl_sync(fullmask, ok, 0);
          if (!ok) break;
          continue;
        }
        if (lane == 0) {
          const uint32_t pb = n % C::kPBufs, pu = n / C::kPBufs;
          if (kPair) {
            // the peer's V half, then both CTAs' P (its softmax warps arrive here)
            mbar_arrive_expect_tx(bar(kPeerV0 + static_cast<int>(s)), 16);  // the peer's V signal
            mbar_arrive_expect_tx(bar(kPFull0 + pb), 16);                    // the peer's P signal
            ok = wait_one_cl(bar(kPeerV0 + static_cast<int>(s)), (n / C::kVStages) & 1u, ctl) &&
                 wait_one_cl(bar(kPFull0 + pb), pu & 1u, ctl);
          } else {
            ok = wait_one(bar(kPFull0 + pb), pu & 1u, ctl);
          }
          if (ok) {
            tc_fence_after();
            const bool first = kt == it.kt0;
            const uint32_t v_lo = desc_lo_at(dv, s * C::kVStage);
            if constexpr (kF8V) {
              // 32 keys (bytes) per MMA; key half hh into its own O
#pragma unroll
              for (int kk = 0; kk < BN / 32; ++kk) {
                const int hh = kk / (BN / 64);
                umma_f8_ts(tmem + C::kColO + hh * D, tmem + C::p_col(static_cast<int>(pb), kk),
                           v_lo + ((kk * 32) >> 4), dv.hi, idesc_pv, (first && kk == hh * (BN / 64)) ? 0u : 1u);
              }
              umma_commit(bar(kVEmpty0 + s));
            }
#pragma unroll
            for (int kk = 0; kk < (kF8V ? 0 : BN / 16); ++kk) {
              const uint32_t b_lo = v_lo + ((kk * (16 * 128)) >> 4);
              const uint32_t a = tmem + C::p_col(static_cast<int>(pb), kk);
              if constexpr (C::kSplitO) {
                // key half hh accumulates into its own O (columns hh * D ...)
                const int hh = kk / (BN / 32);
                umma_f16_ts(tmem + C::kColO + hh * D, a, b_lo, dv.hi, idesc_pv,
                            (first && kk == hh * (BN / 32)) ? 0u : 1u);
              } else if constexpr (kPair) {
                umma_f16_ts_pair(tmem + C::kColO, a, b_lo, dv.hi, idesc_pv, (first && kk == 0) ? 0u : 1u);
              } else {
                umma_f16_ts(tmem + C::kColO, a, b_lo, dv.hi, idesc_pv, (first && kk == 0) ? 0u : 1u);
              }
            }
            // PV of tile n done; its P and V stage are free (in both CTAs of a pair)
            if constexpr (kPair) umma_commit_pair(pv_bar(n));
            else umma_commit(pv_bar(n));
          }
        }
        ok = __shfl_sync(fullmask, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0 && (!kPair || rank == 0)) {
      if constexpr (kPair) umma_commit_pair(bar(kDrainPV));
      else umma_commit(bar(kDrainPV));
      wait_one(bar(kDrainPV), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    if constexpr (C::kSplitO) {
    // ------------------------------------------------------------ softmax, D = 128
    // Warpgroup h (warps 4-7: h = 0, warps 8-11: h = 1) takes keys [h*KH, h*KH + KH)
    // of every tile for all 128 rows, with its own running max, sum and O; the two
    // halves are merged once per item.
    constexpr int KH = BN / 2;
    const int h = (warp - 4) >> 2;
    const int sw = (warp - 4) & 3;        // TMEM lane quarter
    const int r = sw * 32 + lane;         // query row of this thread
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    float2* xml = reinterpret_cast<float2*>(smem + C::kOffX);  // [2 wg][128] (m, l)
    const uint32_t o_own = tmem + lane_base + C::kColO + h * D;
    const int t_local = r / G;
    const int g = r - t_local * G;
    const float c = p.scale_log2;
    uint32_t n = 0, itl = 0;
    uint32_t n_split = 0;  // split items finished (merge handshakes)
    uint32_t n_slice = 0;  // output slices staged by this warpgroup
    bool ok = true;
    // The next item's descriptor and sequence are loaded one item ahead.
    int4 iv_next = cid < n_items ? p.items[cid] : make_int4(0, 0, 0, 0);
    int4 si_next = cid < n_items ? p.seq_info[iv_next.x & kSeqMask] : make_int4(0, 0, 0, 0);
    for (int kq = 0, idx = cid; idx < n_items && ok;
         idx = cta_item(++kq, cid, ncl), ++itl) {
      const Item it = decode_item(iv_next);
      const int4 si = si_next;
      const int idx_next = cta_item(kq + 1, cid, ncl);
      const bool has_next = idx_next < n_items;
      if (has_next) iv_next = p.items[idx_next];
      const int q0 = si.x, ql = si.y, L = si.z;
      const int tok = it.qt * T + t_local;
      const bool valid = (t_local < T) && (tok < ql);
      int lim = 0;  // keys [0, lim) visible to this row
      if (valid) lim = p.causal ? min(L, L - ql + tok + 1) : L;
      const bool warp_live = __any_sync(0xffffffffu, valid) != 0;
      // e4m3 scores: c times the row's Q scale times the K block's scale; the
      // block of this warpgroup's keys of tile kt is kt * (BN / 64) + h
      float cq = c, ksc_next = 1.f;
      if constexpr (kF8) {
        if (valid) cq = c * p.q_scale[static_cast<size_t>(q0 + tok) * p.n_heads_q + it.hk * G + g];
        ksc_next = p.k_scale[(static_cast<size_t>(it.b) * p.nb_max + it.kt0 * C::kPagesPerTile + h) *
                                 p.n_heads_kv + it.hk];
      }
      float m_used = -INFINITY, l = 0.f;
      for (int kt = it.kt0; kt < it.kt1; ++kt, ++n) {
        const uint32_t sb = n % C::kSBufs, su = n / C::kSBufs;
        const uint32_t pb = n % C::kPBufs;
        const bool first = kt == it.kt0;
        if (!(ok = wait_warp(bar(kSFull0 + sb), su & 1u, ctl))) break;
        tc_fence_after();
        uint32_t sr[KH / 32][32];
        if (warp_live) {
#pragma unroll
          for (int j = 0; j < KH / 32; ++j)
            tmem_ld32(tmem + lane_base + C::kColS + sb * BN + h * KH + j * 32, sr[j]);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < KH / 32; ++j) reg_fence(sr[j]);
        }
        if constexpr (!C::kAliasP) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kSFree0 + sb));
        }
        if (kt + 1 == it.kt1 && has_next) si_next = p.seq_info[iv_next.x & kSeqMask];
        float ct = c;
        if constexpr (kF8) {
          ct = cq * ksc_next;
          if (kt + 1 < it.kt1)
            ksc_next = p.k_scale[(static_cast<size_t>(it.b) * p.nb_max + (kt + 1) * C::kPagesPerTile + h) *
                                     p.n_heads_kv + it.hk];
        }

        const int key0 = kt * BN + h * KH;
        const bool full_tile = key0 + KH <= lim;
        const int nv = lim - key0;  // visible keys of this row in the chunk (any sign)
        uint32_t pk[KH / 2];
        if constexpr (kF8V) {
          // e4m3 of p * 2^2 against the running max first. A tile sum of at
          // most 2^8 bounds every code by 2^8 (inside the e4m3 range): then the
          // running max is kept. Otherwise (and on an item's first tile) the tile
          // max decides: O is rescaled if the max grew by more than 6 (log2
          // units), which again bounds every code by 2^(6 + 2), and P is recomputed.
          uint32_t pk8[KH / 4];
          if (warp_live) {
            const float kSumLimit = 256.0f;
            float lt = 0.f;
            bool exact = first || m_used == -INFINITY;
            if (!exact) {
              lt = full_tile ? exp_row_f8<KH, false>(sr, ct, m_used - 2.0f, KH, pk8)
                             : exp_row_f8<KH, true>(sr, ct, m_used - 2.0f, nv, pk8);
              exact = !(lt <= kSumLimit);  // also true for inf / NaN
            }
            if (__any_sync(0xffffffffu, exact)) {
              const float mx = full_tile ? max_row<KH, false>(sr, KH) : max_row<KH, true>(sr, nv);
              const float mx_s = (mx == -INFINITY) ? -INFINITY : mx * ct;
              const float m_new = fmaxf(m_used, mx_s);
              if (first) {
                m_used = m_new;
              } else {
                const bool need = m_new > m_used + 6.0f;
                if (__any_sync(0xffffffffu, need)) {
                  const uint32_t pm = n - 1;
                  if (!(ok = wait_warp(pv_bar(pm), pv_par(pm), ctl))) break;
                  tc_fence_after();
                  const float alpha = need ? ex2(m_used - m_new) : 1.0f;
                  if (need) {
                    l *= alpha;
                    m_used = m_new;
                  }
#pragma unroll 1
                  for (int j = 0; j < D / 32; ++j) {
                    uint32_t o[32];
                    tmem_ld32(o_own + j * 32, o);
                    tmem_wait_ld();
                    reg_fence(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(o_own + j * 32, o);
                  }
                  tmem_wait_st();
                }
              }
              const float m_ref = ((m_used == -INFINITY) ? 0.f : m_used) - 2.0f;
              lt = full_tile ? exp_row_f8<KH, false>(sr, ct, m_ref, KH, pk8)
                             : exp_row_f8<KH, true>(sr, ct, m_ref, nv, pk8);
            }
            l += lt;
          }
          // P over the S columns this warp has just read (nothing to wait for)
          if (warp_live) {
            tmem_st_cols<KH / 4>(tmem + lane_base + C::p_col(static_cast<int>(pb), h * (BN / 64)), pk8);
            tmem_wait_st();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kPFull0 + pb));
          continue;
        }
        if (warp_live) {
          // Probabilities against the running max first. Their sum bounds every
          // one of them, so a sum of at most 2^8 shows that the tile max exceeds
          // the running max by at most 8 (log2 units): exactly the case in which
          // the running max is kept, and nothing more is needed. Otherwise (and
          // on an item's first tile) the tile max decides, as it always would.
          const float kSumLimit = 256.0f;
          float lt = 0.f;
          bool exact = first || m_used == -INFINITY;
          if (!exact) {
            lt = full_tile ? exp_row<KH, false>(sr, ct, m_used, KH, pk)
                           : exp_row<KH, true>(sr, ct, m_used, nv, pk);
            exact = !(lt <= kSumLimit);  // also true for inf / NaN
          }
          if (__any_sync(0xffffffffu, exact)) {
            float acc[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) acc[u] = -INFINITY;
            if (full_tile) {
#pragma unroll
              for (int j = 0; j < KH / 32; ++j)
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[i & 7] = fmaxf(acc[i & 7], __uint_as_float(sr[j][i]));
            } else {
#pragma unroll
              for (int j = 0; j < KH / 32; ++j)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (j * 32 + i < nv) acc[i & 7] = fmaxf(acc[i & 7], __uint_as_float(sr[j][i]));
            }
            const float mx = fmaxf(fmaxf(fmaxf(acc[0], acc[1]), fmaxf(acc[2], acc[3])),
                                   fmaxf(fmaxf(acc[4], acc[5]), fmaxf(acc[6], acc[7])));
            const float mx_s = (mx == -INFINITY) ? -INFINITY : mx * ct;
            const float m_new = fmaxf(m_used, mx_s);
            if (first) {
              m_used = m_new;
            } else {
              const bool need = m_new > m_used + 8.0f;
              if (__any_sync(0xffffffffu, need)) {
                // this half's O holds the previous tiles; rescale it once their PV is done
                const uint32_t pm = n - 1;
                if (!(ok = wait_warp(pv_bar(pm), pv_par(pm), ctl))) break;
                tc_fence_after();
                const float alpha = need ? ex2(m_used - m_new) : 1.0f;
                if (need) {
                  l *= alpha;
                  m_used = m_new;
                }
#pragma unroll 1
                for (int j = 0; j < D / 32; ++j) {
                  uint32_t o[32];
                  tmem_ld32(o_own + j * 32, o);
                  tmem_wait_ld();
                  reg_fence(o);
#pragma unroll
                  for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                  tmem_st32(o_own + j * 32, o);
                }
                tmem_wait_st();
              }
            }
            const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
            lt = full_tile ? exp_row<KH, false>(sr, ct, m_ref, KH, pk)
                           : exp_row<KH, true>(sr, ct, m_ref, nv, pk);
          }
          l += lt;
        }
        // P buffer pb was last read by the PV of tile n - kPBufs (written over S:
        // the columns this warp has just read, nothing to wait for)
        if (!C::kAliasP && n >= static_cast<uint32_t>(C::kPBufs)) {
          const uint32_t pm = n - C::kPBufs;
          if (!(ok = wait_warp(pv_bar(pm), pv_par(pm), ctl))) break;
        }
        if (warp_live) {
          tmem_st_cols<KH / 2>(tmem + lane_base + C::p_col(static_cast<int>(pb), h * (BN / 32)), pk);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kPFull0 + pb));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue: merge the halves
      xml[h * kBM + r] = make_float2(m_used, l);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kXSum));
      if (!(ok = wait_warp(bar(kXSum), itl & 1u, ctl))) break;
      const float2 a0 = xml[r], a1 = xml[kBM + r];
      const float M = fmaxf(a0.x, a1.x);
      const float w0 = a0.y > 0.f ? ex2(a0.x - M) : 0.f;
      const float w1 = a1.y > 0.f ? ex2(a1.x - M) : 0.f;
      const float den = w0 * a0.y + w1 * a1.y;
      const float inv = den > 0.f ? 1.0f / den : 0.f;
      const float c0 = w0 * inv, c1 = w1 * inv;
      {
        const uint32_t pm = n - 1;
        if (!(ok = wait_warp(pv_bar(pm), pv_par(pm), ctl))) break;
      }
      tc_fence_after();
      // An unsplit item whose q tile is full leaves through the tensor store:
      // each warpgroup stages a 32-column slice of its 128 rows and one thread
      // stores the box [32 channels, G heads, 1, T tokens] (whole 64-byte row
      // pieces instead of 16 bytes per thread and row). The other items store
      // row by row below.
      const bool tma_out = it.part < 0 && (it.qt + 1) * T <= ql;
      if (tma_out) {
        // (bounded mbarrier hand-offs, not a named barrier: a warp that gave up
        // elsewhere cannot leave the others of its warpgroup waiting)
        const uint32_t stage = s_base + C::kOffO + static_cast<uint32_t>(h * (kBM * 64));
        const uint32_t row_addr = stage + static_cast<uint32_t>(r * 64);
        const uint32_t sx = static_cast<uint32_t>((r >> 1) & 3);  // 64-byte swizzle of this row
#pragma unroll 1
        for (int pp = 0; pp < 2 && ok; ++pp, ++n_slice) {
          const int col = h * (D / 2) + pp * 32;
          // the slice buffer is free once the previous store has read it
          if (!(ok = wait_warp(bar(kOSlFree0 + h), (n_slice & 1u) ^ 1u, ctl))) break;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int cc = col + hf * 16;
            float4 vsc[4];
            if constexpr (kF8V) {
              // per-channel V scale (P's 2^2 cancels against l)
              const float4* vs = reinterpret_cast<const float4*>(
                  p.v_scale + (static_cast<size_t>(it.b) * p.n_heads_kv + it.hk) * D + cc);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) vsc[q4] = vs[q4];
            }
            uint32_t o0[16], o1[16];
            tmem_ld16(tmem + lane_base + C::kColO + cc, o0);
            tmem_ld16(tmem + lane_base + C::kColO + D + cc, o1);
            tmem_wait_ld();
            reg_fence(o0);
            reg_fence(o1);
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              float a = __uint_as_float(o0[2 * e]) * c0 + __uint_as_float(o1[2 * e]) * c1;
              float b = __uint_as_float(o0[2 * e + 1]) * c0 + __uint_as_float(o1[2 * e + 1]) * c1;
              if constexpr (kF8V) {
                const float4 f = vsc[e >> 1];
                a *= (e & 1) ? f.z : f.x;
                b *= (e & 1) ? f.w : f.y;
              }
              __nv_bfloat162 hh = __floats2bfloat162_rn(a, b);
              w[e] = *reinterpret_cast<uint32_t*>(&hh);
            }
            // 16-byte chunks 2 hf and 2 hf + 1 of the row, swizzled
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
              st_shared_v4(row_addr + ((static_cast<uint32_t>(2 * hf + c2) ^ sx) << 4), w[4 * c2],
                           w[4 * c2 + 1], w[4 * c2 + 2], w[4 * c2 + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kOSlFull0 + h));
          if (sw == 0) {
            if (lane == 0) {
              ok = wait_one(bar(kOSlFull0 + h), n_slice & 1u, ctl);
              if (ok) {
                tma_store_4d(&tmap_o, stage, col, 0, it.hk, q0 + it.qt * T);
                bulk_commit_group();
                bulk_wait_read_all();
                mbar_arrive(bar(kOSlFree0 + h));
              }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
          }
        }
        if (!ok) break;
      } else if (warp_live) {
        const int hq = it.hk * G + g;
#pragma unroll 1
        for (int j = 0; j < (D / 2) / 16; ++j) {
          const int col = h * (D / 2) + j * 16;  // this warpgroup writes half of the columns
          uint32_t o0[16], o1[16];
          tmem_ld16(tmem + lane_base + C::kColO + col, o0);
          tmem_ld16(tmem + lane_base + C::kColO + D + col, o1);
          tmem_wait_ld();
          reg_fence(o0);
          reg_fence(o1);
          if (!valid) continue;
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(o0[i]) * c0 + __uint_as_float(o1[i]) * c1;
          if constexpr (kF8V) {
            // per-channel V scale (P's 2^2 cancels against l)
            const float4* vs = reinterpret_cast<const float4*>(
                p.v_scale + (static_cast<size_t>(it.b) * p.n_heads_kv + it.hk) * D + col);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const float4 f = vs[q4];
              v[q4 * 4] *= f.x;
              v[q4 * 4 + 1] *= f.y;
              v[q4 * 4 + 2] *= f.z;
              v[q4 * 4 + 3] *= f.w;
            }
          }
          if (it.part < 0) {
            uint4* dst = reinterpret_cast<uint4*>(
                p.out + (static_cast<size_t>(q0 + tok) * p.n_heads_q + hq) * D + col);
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
            float4* dst = reinterpret_cast<float4*>(p.part_o + static_cast<size_t>(it.part + r) * D + col);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              dst[q4] = make_float4(v[q4 * 4], v[q4 * 4 + 1], v[q4 * 4 + 2], v[q4 * 4 + 3]);
          }
        }
        if (valid && it.part >= 0 && h == 0)
          p.part_ml[it.part + r] = make_float2(den > 0.f ? M : -INFINITY, den);
      }
      tc_fence_before();
      if (it.part >= 0 &&
          !(ok = split_done<D>(p, it, si, bar(kMergeA), bar(kMergeB), merge_flag, n_split, warp, ctl)))
        break;
    }
    // the output stores of this warpgroup complete before the CTA exits
    if (sw == 0 && lane == 0) bulk_wait_all();
    } else {
    // ------------------------------------------------------------ softmax: two warpgroups
    // Warpgroup h (warps 4-7: h = 0, warps 8-11: h = 1) takes keys [h*KH, h*KH + KH)
    // of every tile and O columns [h*DH, h*DH + DH) for the same 128 rows. Warp w
    // and warp w + 4 hold the same 32 rows: they exchange their partial row sums
    // once per tile (and their partial row maxes when those are needed).
    constexpr int KH = BN / 2;
    constexpr int DH = D / 2;
    const int h = (warp - 4) >> 2;
    const int sw = (warp - 4) & 3;        // TMEM lane quarter
    const int r = sw * 32 + lane;         // query row of this thread
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    float* xsum_t = reinterpret_cast<float*>(smem + C::kOffX);  // [2 parity][2 wg][128]
    float* xmax_t = xsum_t + 2 * 2 * kBM;                         // [2 parity][2 wg][128]
    float* xl = xmax_t + 2 * 2 * kBM;                             // [2 wg][128]
    const uint32_t pair_a = bar(kPairA0 + sw), pair_b = bar(kPairB0 + sw);
    const int t_local = r / G;
    const int g = r - t_local * G;
    const float c = p.scale_log2;
    const float kSumLimit = 256.0f;  // 2^8: the running max is kept while every p <= 2^8
    const unsigned full = 0xffffffffu;
    uint32_t n = 0, itl = 0;
    uint32_t n_split = 0;  // split items finished (merge handshakes)
    uint32_t na = 0, nb = 0;  // row-sum / row-max exchanges of this warp pair
    bool ok = true;
    int4 iv_next = cid < n_items ? p.items[cid] : make_int4(0, 0, 0, 0);
    int4 si_next = cid < n_items ? p.seq_info[iv_next.x & kSeqMask] : make_int4(0, 0, 0, 0);
    for (int kq = 0, idx = cid; idx < n_items && ok;
         idx = cta_item(++kq, cid, ncl), ++itl) {
      const Item it = decode_item(iv_next);
      const int4 si = si_next;
      const int idx_next = cta_item(kq + 1, cid, ncl);
      const bool has_next = idx_next < n_items;
      if (has_next) iv_next = p.items[idx_next];
      const int q0 = si.x, ql = si.y, L = si.z;
      const int tok = (it.qt + static_cast<int>(rank)) * T + t_local;  // a pair's peer: the next q tile
      const bool valid = (t_local < T) && (tok < ql);
      int lim = 0;  // keys [0, lim) visible to this row
      if (valid) lim = p.causal ? min(L, L - ql + tok + 1) : L;
      // the same for both warps of a pair (same rows)
      const bool warp_live = __any_sync(full, valid) != 0;
      float m_used = -INFINITY, l = 0.f;
      for (int kt = it.kt0; kt < it.kt1; ++kt, ++n) {
        const uint32_t sb = n % C::kSBufs, pb = n % C::kPBufs;
        const bool first = kt == it.kt0;
        if (!(ok = wait_warp(bar(kSFull0 + sb), (n / C::kSBufs) & 1u, ctl))) break;
        tc_fence_after();
        uint32_t sr[KH / 32][32];
        if (warp_live) {
#pragma unroll
          for (int j = 0; j < KH / 32; ++j)
            tmem_ld32(tmem + lane_base + C::kColS + sb * BN + h * KH + j * 32, sr[j]);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < KH / 32; ++j) reg_fence(sr[j]);
        }
        if constexpr (!C::kAliasP) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kSFree0 + sb));
        }
        if (kt + 1 == it.kt1 && has_next) si_next = p.seq_info[iv_next.x & kSeqMask];
        // a separate P buffer was last read by the PV of tile n - kPBufs; over S,
        // P goes into the columns this warp has just read
        if (!C::kAliasP && n >= static_cast<uint32_t>(C::kPBufs)) {
          if (!(ok = wait_warp(pv_bar(n - C::kPBufs), pv_par(n - C::kPBufs), ctl))) break;
        }
        const int key0 = kt * BN + h * KH;
        const bool full_tile = key0 + KH <= lim;
        const int nv = lim - key0;  // visible keys of this row in the chunk (any sign)
        const uint32_t p_addr = tmem + lane_base + C::p_col(static_cast<int>(pb), h * (BN / 32));
        uint32_t pk[KH / 2];
        float lt = 0.f;
        if (warp_live) {
          bool exact = first;
          if (!first) {
            // P against the running max; a row that has seen no key yet (m = -inf)
            // takes the exact path if it sees one now
            const float m_spec = m_used == -INFINITY ? 0.f : m_used;
            lt = full_tile ? exp_row<KH, false>(sr, c, m_spec, KH, pk)
                           : exp_row<KH, true>(sr, c, m_spec, nv, pk);
            tmem_st_cols<KH / 2>(p_addr, pk);
            // round A: the row's two half sums (+inf forces the exact path)
            xsum_t[((na & 1u) * 2 + h) * kBM + r] = (m_used == -INFINITY && nv > 0) ? INFINITY : lt;
            __syncwarp();
            if (lane == 0) mbar_arrive(pair_a);
            if (!(ok = wait_warp(pair_a, na & 1u, ctl))) break;
            const float mine = xsum_t[((na & 1u) * 2 + h) * kBM + r];
            const float tot = mine + xsum_t[((na & 1u) * 2 + (1 - h)) * kBM + r];
            ++na;
            exact = !(tot <= kSumLimit);  // also true for inf / NaN
          }
          if (__any_sync(full, exact)) {
            // round B: the tile max of the row over both halves
            float mx = full_tile ? max_row<KH, false>(sr, nv) : max_row<KH, true>(sr, nv);
            xmax_t[((nb & 1u) * 2 + h) * kBM + r] = mx;
            __syncwarp();
            if (lane == 0) mbar_arrive(pair_b);
            if (!(ok = wait_warp(pair_b, nb & 1u, ctl))) break;
            mx = fmaxf(mx, xmax_t[((nb & 1u) * 2 + (1 - h)) * kBM + r]);
            ++nb;
            const float mx_s = (mx == -INFINITY) ? -INFINITY : mx * c;
            const float m_new = fmaxf(m_used, mx_s);
            if (first) {
              m_used = m_new;
            } else {
              const bool need = m_new > m_used + 8.0f;
              if (__any_sync(full, need)) {
                // O holds the previous tiles; rescale this warpgroup's half of the
                // columns once their PV is done
                if (!(ok = wait_warp(pv_bar(n - 1), pv_par(n - 1), ctl))) break;
                tc_fence_after();
                const float alpha = need ? ex2(m_used - m_new) : 1.0f;
                if (need) {
                  l *= alpha;
                  m_used = m_new;
                }
#pragma unroll 1
                for (int j = 0; j < DH / 32; ++j) {
                  uint32_t o[32];
                  tmem_ld32(tmem + lane_base + C::kColO + h * DH + j * 32, o);
                  tmem_wait_ld();
                  reg_fence(o);
#pragma unroll
                  for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                  tmem_st32(tmem + lane_base + C::kColO + h * DH + j * 32, o);
                }
              }
            }
            const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
            lt = full_tile ? exp_row<KH, false>(sr, c, m_ref, KH, pk)
                           : exp_row<KH, true>(sr, c, m_ref, nv, pk);
            tmem_wait_st();  // the speculative P (if any) lands before it is overwritten
            tmem_st_cols<KH / 2>(p_addr, pk);
          }
          l += lt;
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kPFull0 + pb));  // (a pair's peer forwards it from warp 2)
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      xl[h * kBM + r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kXSum));
      if (!(ok = wait_warp(bar(kXSum), itl & 1u, ctl))) break;
      const float l_all = l + xl[(1 - h) * kBM + r];
      if (!(ok = wait_warp(pv_bar(n - 1), pv_par(n - 1), ctl))) break;
      tc_fence_after();
      if (warp_live) {
        const float inv_l = l_all > 0.f ? 1.0f / l_all : 0.f;
        const int hq = it.hk * G + g;
#pragma unroll 1
        for (int j = 0; j < DH / 32; ++j) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + C::kColO + h * DH + j * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          if (!valid) continue;
          const int col = h * DH + j * 32;
          if (it.part < 0) {
            uint4* dst = reinterpret_cast<uint4*>(
                p.out + (static_cast<size_t>(q0 + tok) * p.n_heads_q + hq) * D + col);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 hh = __floats2bfloat162_rn(__uint_as_float(o[v * 8 + 2 * e]) * inv_l,
                                                          __uint_as_float(o[v * 8 + 2 * e + 1]) * inv_l);
                w[e] = *reinterpret_cast<uint32_t*>(&hh);
              }
              dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(
                p.part_o + static_cast<size_t>(it.part + r) * D + col);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(o[v * 4]) * inv_l, __uint_as_float(o[v * 4 + 1]) * inv_l,
                                   __uint_as_float(o[v * 4 + 2]) * inv_l,
                                   __uint_as_float(o[v * 4 + 3]) * inv_l);
          }
        }
        if (valid && it.part >= 0 && h == 0)
          p.part_ml[it.part + r] = make_float2(l_all > 0.f ? m_used : -INFINITY, l_all);
      }
      tc_fence_before();
      // (a pair's peer holds no rows of a split item: single-q-tile units only)
      if (it.part >= 0 && (!kPair || rank == 0) &&
          !(ok = split_done<D>(p, it, si, bar(kMergeA), bar(kMergeB), merge_flag, n_split, warp, ctl)))
        break;
    }
    }
  }

  tc_fence_before();
  __syncthreads();
  // a pair leaves together: no cross-CTA arrive or MMA targets a CTA that has left
  if constexpr (kPair) cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (kPair) tmem_dealloc_pair(tmem, kTmemCols);
    else tmem_dealloc(tmem, kTmemCols);
  }
  prefill_end(p);
}

}  // namespace

int attention_block_n(int head_dim, bool pair) { return head_dim == 128 || pair ? 128 : 64; }

size_t attention_smem_bytes(int head_dim) {
  return head_dim == 128 ? static_cast<size_t>(Cfg<128, 128>::kSmem)
                         : static_cast<size_t>(Cfg<256, 64>::kSmem);
}

cudaError_t attention_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<128, 128, false, false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<128, 128>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_kernel<128, 128, true, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128, 128, true>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_kernel<128, 128, true, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128, 128, true, true>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_kernel<256, 128, false, false, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<256, 128, false, false, true>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_kernel<256, 64, false, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<256, 64>::kSmem);
}

cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tkv,
                             const CUtensorMap& to, int head_dim, int grid, cudaStream_t s, bool dependent) {
  if (head_dim == 128)
    return launch_kernel(attn_kernel<128, 128, false, false, false>, grid, kAttnThreads, Cfg<128, 128>::kSmem, s,
                         dependent, tq, tkv, tkv, tkv, to, p);
  return launch_kernel(attn_kernel<256, 64, false, false, false>, grid, kAttnThreads, Cfg<256, 64>::kSmem, s,
                       dependent, tq, tkv, tkv, tkv, tq, p);
}

cudaError_t launch_attention_fp8(const AttnParams& p, const CUtensorMap& tq8, const CUtensorMap& tk8,
                                 const CUtensorMap& tkv, const CUtensorMap& to, int grid, cudaStream_t s,
                                 bool dependent) {
  return launch_kernel(attn_kernel<128, 128, true, false, false>, grid, kAttnThreads, Cfg<128, 128, true>::kSmem,
                       s, dependent, tq8, tkv, tk8, tkv, to, p);
}

cudaError_t launch_attention_fp8pv(const AttnParams& p, const CUtensorMap& tq8, const CUtensorMap& tk8,
                                   const CUtensorMap& tv8, const CUtensorMap& to, int grid, cudaStream_t s,
                                   bool dependent) {
  return launch_kernel(attn_kernel<128, 128, true, true, false>, grid, kAttnThreads,
                       Cfg<128, 128, true, true>::kSmem, s, dependent, tq8, tv8, tk8, tv8, to, p);
}

cudaError_t launch_attention_pair(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tkv,
                                  int grid, cudaStream_t s, bool dependent) {
  return launch_kernel_pair(attn_kernel<256, 128, false, false, true>, grid & ~1, kAttnThreads,
                            Cfg<256, 128, false, false, true>::kSmem, s, dependent, tq, tkv, tkv, tkv, tq, p);
}

}  // namespace pattn
