// plan.cu -- device-side varlen tile scheduler.
//
// plan_kernel (one CTA) turns (cu_q, seq_lens, block_table) into the work list
// the attention kernel walks, without a host round trip:
//   1. validates every sequence (query range inside [0, total_q], lengths within
//      the host bounds, every live block-table entry inside the pool); a
//      rejected sequence sets the device error word and gets zero output;
//   2. cuts each sequence into q tiles of T = 128 / G tokens (GQA packing) and,
//      per q tile, keeps only the KV tiles the causal mask leaves visible
//      (tiles wholly above the diagonal are never scheduled, the "fully
//      masked" status of the FlashAttention-4 kernel doc's mask_status);
//   3. splits the KV range of single-q-tile units (decode) so that each
//      kernel's list (the decode kernel's, the prefill kernel's: they run one
//      after the other) has about `target_items` items of at least `min_chunk`
//      tiles of its own work (the
//      decode manifest's "MultiCtasKv": several CTAs per sequence and KV
//      head, with partial O and (max, sum) statistics in scratch). When the
//      decode units' lengths are skewed (the longest more than 2.5 times the
//      mean), the decode list's target is chosen per call between
//      target_items and 1.25 x target_items: the one whose items give the
//      smaller largest CTA load under the decode kernel's item order (a
//      counting sort of the item costs and the alternating round robin,
//      simulated per CTA);
//   4. orders the items longest first (counting sort on the number of KV
//      tiles) so that round-robin assignment to persistent CTAs balances;
//   5. zero-fills the output rows of q tiles that see no key at all, and
//      zeroes the finished-split counter of every split unit (the attention
//      kernels merge a unit's partials in the CTA that finishes it last).
//
// With new tokens to cache (pattn_forward_append), the grid has more CTAs:
// while CTA 0 plans, the others write the new tokens' K and V rows into their
// cache slots, the `reshape_and_cache_flash` (kv_write) node that comes right
// before `attend` in the GB10 model graph. The attention kernels wait for the
// whole plan grid, so they read the updated cache, and no launch of its own
// is spent on the write.
#include <algorithm>

#include "kernels.cuh"
#include "ptx.cuh"

namespace pattn {
namespace {

// Threads of the planning CTA: 1024 for large batches; small batches (few
// sequences and q tiles) plan faster on 128, since every phase of the plan is
// a block-wide step whose cost grows with the warps that take part.
constexpr int kPlanThreads = 1024;
constexpr int kPlanThreadsSmall = 128;
constexpr int kPlanSmallSeqs = 32;  // batches of at most this many sequences take the small CTA

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Hint: bring the 128-byte line holding `ptr` into L2 (no value is read; a
// later load sees whatever was written there meanwhile).
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(ptr)));
}

// Units of at most kDecRows packed rows run on the swap-AB decode kernel.
__device__ __forceinline__ bool is_decode(const PlanParams& p, int ql) {
  return p.dec_enabled && ql >= 1 && ql * p.group <= kDecRows;
}

// log2 of the keys per KV tile of the kernel a unit of ql queries goes to (the
// tile sizes are powers of two, so tile counts are shifts, not divisions).
__device__ __forceinline__ int tile_shift(const PlanParams& p, int ql) {
  return is_decode(p, ql) ? kDecBlockNShift : p.block_n_shift;
}

// Visible KV tiles of q tile qt: keys [0, kv_hi), kv_hi the largest limit of its rows.
__device__ __forceinline__ int qtile_kv_tiles(const PlanParams& p, int ql, int L, int qt) {
  int hi = L;
  if (p.causal) {
    const int last_tok = min(ql, (qt + 1) * p.tokens_per_tile);
    hi = min(L, L - ql + last_tok);
  }
  const int sh = tile_shift(p, ql);
  return hi > 0 ? (hi + (1 << sh) - 1) >> sh : 0;
}

// Work of a q tile in 64-key blocks (comparable across the two kernels' tile sizes).
__device__ __forceinline__ int qtile_blocks(const PlanParams& p, int ql, int L, int qt) {
  return qtile_kv_tiles(p, ql, L, qt) << (tile_shift(p, ql) - kPageShift);
}

// Warp sum of a 64-bit count: two single-instruction 32-bit reductions when
// every lane's value fits 32 bits (the usual case), else a shuffle tree.
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
  const unsigned full = 0xffffffffu;
  if (!__any_sync(full, (v >> 32) != 0ull)) {
    const unsigned hi = __reduce_add_sync(full, static_cast<unsigned>(v >> 8));
    const unsigned lo = __reduce_add_sync(full, static_cast<unsigned>(v & 255ull));
    return (static_cast<unsigned long long>(hi) << 8) + lo;
  }
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(full, v, o);
  return v;
}

// Block-wide exclusive scan of two ints per thread (NT threads); returns both block totals.
template <int NT>
__device__ int2 block_exclusive_scan2(int v0, int v1, int* e0, int* e1, int2* warp_sums) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x0 = v0, x1 = v1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y0 = __shfl_up_sync(0xffffffffu, x0, o);
    const int y1 = __shfl_up_sync(0xffffffffu, x1, o);
    if (lane >= o) {
      x0 += y0;
      x1 += y1;
    }
  }
  if (lane == 31) warp_sums[warp] = make_int2(x0, x1);
  __syncthreads();
  if (warp == 0) {
    int2 w = lane < kWarps ? warp_sums[lane] : make_int2(0, 0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y0 = __shfl_up_sync(0xffffffffu, w.x, o);
      const int y1 = __shfl_up_sync(0xffffffffu, w.y, o);
      if (lane >= o) {
        w.x += y0;
        w.y += y1;
      }
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const int2 before = warp ? warp_sums[warp - 1] : make_int2(0, 0);
  *e0 = before.x + x0 - v0;
  *e1 = before.y + x1 - v1;
  const int2 total = warp_sums[kWarps - 1];
  __syncthreads();
  return total;
}

// Exclusive starts of both item lists' histograms, from the most expensive
// bucket down (a counting sort, longest first); returns the list totals. Each
// thread takes kHistBuckets / NT consecutive buckets.
template <int NT>
__device__ int2 scan_hist_desc(int (*hist)[kHistBuckets], int2* warp_sums) {
  static_assert(kHistBuckets % NT == 0, "whole buckets per thread");
  constexpr int R = kHistBuckets / NT;
  const int c0 = kHistBuckets - 1 - static_cast<int>(threadIdx.x) * R;  // buckets c0, c0 - 1, ..
  int v0[R], v1[R], s0 = 0, s1 = 0;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    v0[i] = hist[0][c0 - i];
    v1[i] = hist[1][c0 - i];
    s0 += v0[i];
    s1 += v1[i];
  }
  int e0, e1;
  const int2 tot = block_exclusive_scan2<NT>(s0, s1, &e0, &e1, warp_sums);
#pragma unroll
  for (int i = 0; i < R; ++i) {
    hist[0][c0 - i] = e0;
    hist[1][c0 - i] = e1;
    e0 += v0[i];
    e1 += v1[i];
  }
  return tot;
}

// Work of all q tiles of a sequence in 64-key blocks, for the split heuristic
// only: exact for short sequences, an arithmetic-series estimate for long ones.
__device__ __forceinline__ unsigned long long seq_blocks(const PlanParams& p, int ql, int L, int nqt) {
  if (nqt <= 8) {
    unsigned long long t = 0;
    for (int qt = 0; qt < nqt; ++qt) t += static_cast<unsigned long long>(qtile_blocks(p, ql, L, qt));
    return t;
  }
  const int sh = tile_shift(p, ql);
  if (!p.causal)
    return static_cast<unsigned long long>(nqt) * (((L + (1 << sh) - 1) >> sh) << (sh - kPageShift));
  // keys [0, L - ql + (qt + 1) T) for qt < nqt - 1, keys [0, L) for the last q tile
  const long long T = p.tokens_per_tile;
  const long long n1 = nqt - 1;
  const long long keys = max(n1 * (static_cast<long long>(L) - ql) + T * n1 * (n1 + 1) / 2 + L, 0ll);
  return static_cast<unsigned long long>((keys >> kPageShift) + (static_cast<long long>(nqt) << (sh - kPageShift)) / 2 + 1);
}

// ---- cache write of the new tokens ----------------------------------------
// Token i of sequence b (i < ql_b) is cache position L_b - ql_b + i, the same
// bottom-right alignment the attention uses: slot pos / 64 of the block table
// and row pos % 64 of that page, or row pos of the sequence in a contiguous
// cache. A sequence the planner rejects is not written, so each writing warp
// applies the planner's acceptance rules to the sequences of its tokens
// itself (it cannot wait for CTA 0): query range inside [0, total_q] with
// ql <= max_q, 0 <= L <= max_kv, and every live block-table entry inside the
// pool (paged) or the sequence's rows inside the K/V planes (contiguous).
struct SeqCheck {
  int q0, q1, L;
  long long row0;  // first row of the sequence in a contiguous cache
  bool ok;
};

// One warp, same result in every lane.
__device__ SeqCheck warp_check_seq(const PlanParams& p, int b) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  SeqCheck c;
  c.q0 = p.cu_q[b];
  c.q1 = p.cu_q[b + 1];
  c.L = p.seq_lens[b];
  c.row0 = 0;
  c.ok = c.q0 >= 0 && c.q1 >= c.q0 && c.q1 <= p.total_q && c.q1 - c.q0 <= p.max_q && c.L >= 0 &&
         c.L <= p.max_kv;
  if (!c.ok) return c;
  if (p.block_table) {
    const int np = cdiv(c.L, kPage);
    const int32_t* row = p.block_table + static_cast<size_t>(b) * p.bt_stride;
    bool bad = false;
    for (int s = lane; s < np; s += 32) {
      const int pg = row[s];
      bad |= pg < 0 || pg >= p.num_pages;
    }
    c.ok = !__any_sync(full, bad);
  } else {
    // rows of the sequences before b (negative lengths count as zero, as in the plan)
    long long sum = 0;
    for (int i = lane; i < b; i += 32) sum += max(p.seq_lens[i], 0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(full, sum, o);
    c.row0 = sum;
    c.ok = sum + c.L <= static_cast<long long>(p.num_pages);
  }
  return c;
}

// CTAs 1.. of the plan grid: one warp per run of consecutive tokens; each
// token's K row and V row ([Hkv][D] each, contiguous) are copied with 16-byte
// streaming loads, all loads of a chunk issued before its stores.
__device__ void write_new_rows(const PlanParams& p) {
  const int lane = threadIdx.x & 31;
  const int per_cta = static_cast<int>(blockDim.x) >> 5;
  const int warps = (static_cast<int>(gridDim.x) - 1) * per_cta;
  const int w = (static_cast<int>(blockIdx.x) - 1) * per_cta + (threadIdx.x >> 5);
  const int per = cdiv(p.total_q, warps);
  const int t0 = w * per, t1 = min(p.total_q, t0 + per);
  if (t0 >= t1) return;
  // sequence of token t0: the last b with cu_q[b] <= t0 (each sequence found is
  // checked below, so an out-of-order cu_q writes nothing)
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu_q[mid] <= t0) lo = mid; else hi = mid - 1;
  }
  int b = lo, checked = -1;
  SeqCheck c{};
  const int row_elems = p.n_heads_kv * p.head_dim;
  const int n16 = row_elems / 8;  // 16-byte chunks of one token's K (or V) row
  for (int t = t0; t < t1; ++t) {
    while (b + 1 < p.num_seqs && p.cu_q[b + 1] <= t) ++b;
    if (b != checked) {
      c = warp_check_seq(p, b);
      checked = b;
    }
    if (!c.ok || t < c.q0 || t >= c.q1) continue;
    const int pos = c.L - (c.q1 - c.q0) + (t - c.q0);
    if (pos < 0) continue;  // more queries than keys: no slot for this token
    size_t krow, vrow;      // element offsets of the destination rows
    if (p.block_table) {
      const int page = p.block_table[static_cast<size_t>(b) * p.bt_stride + pos / kPage];
      krow = (static_cast<size_t>(page) * 2 * kPage + (pos % kPage)) * row_elems;
      vrow = krow + static_cast<size_t>(kPage) * row_elems;
    } else {
      krow = static_cast<size_t>(c.row0 + pos) * row_elems;
      vrow = krow + static_cast<size_t>(p.num_pages) * row_elems;
    }
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_new + static_cast<size_t>(t) * row_elems);
    const uint4* vs = reinterpret_cast<const uint4*>(p.v_new + static_cast<size_t>(t) * row_elems);
    uint4* kd = reinterpret_cast<uint4*>(p.kv_pool + krow);
    uint4* vd = reinterpret_cast<uint4*>(p.kv_pool + vrow);
    for (int j0 = 0; j0 < n16; j0 += 4 * 32) {
      uint4 kv[4], vv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * 32 + lane;
        if (j < n16) {
          kv[u] = __ldcs(ks + j);
          vv[u] = __ldcs(vs + j);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * 32 + lane;
        if (j < n16) {
          kd[j] = kv[u];
          vd[j] = vv[u];
        }
      }
    }
  }
}

// Balance model of the decode list's split target: each item costs its KV
// tiles plus kItemCost tiles (pipeline fill and drain, epilogue, split
// merge). The choice is simulated only for skewed lengths (longest unit more
// than 2.5 times the mean; equal-length units balance at the base target) and
// for at most kBalanceUnitsPerCta units per CTA (the simulation walks every
// CTA's items).
constexpr int kItemCost = 2;
constexpr int kBalanceUnitsPerCta = 4;

constexpr int kSmemSeqs = 4096;   // sequences whose q-tile prefix is kept in shared memory
constexpr int kCacheSeqs = 1024;  // sequences whose plan is kept in shared memory

template <int NT>
__global__ void __launch_bounds__(NT, 1) plan_kernel(const PlanParams p) {
  __shared__ int2 warp_sums[32];
  __shared__ int hist[2][kHistBuckets];  // [0] prefill items, [1] decode items
  __shared__ int s_qt_prefix[kSmemSeqs];
  __shared__ int4 s_seq[kCacheSeqs];     // x = first token, y = query length (-1 rejected), z = L, w = splits
  __shared__ int s_part[kCacheSeqs];     // first partial row of the sequence's split units
  __shared__ int s_carry[4];
  __shared__ unsigned long long s_tiles[2];  // work of the prefill [0] and decode [1] kernels
  __shared__ int s_list_items[2];
  __shared__ int s_need_zero;     // some sequence is rejected or has q tiles that see no key
  __shared__ int s_dec_units;     // decode sequences
  __shared__ int s_dec_max;       // KV tiles of the longest decode unit
  __shared__ int s_load[2];       // largest CTA load under each candidate target
  const Workspace& ws = p.ws;
  const int B = p.num_seqs;
  const int G = p.group;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto seq_at = [&](int b) -> int4 {
    if (b < kCacheSeqs) return s_seq[b];
    const int4 si = ws.seq_info[b];
    return make_int4(si.x, si.y, si.z, ws.seq_plan[b].z);
  };
  auto part_at = [&](int b) -> int { return b < kCacheSeqs ? s_part[b] : ws.seq_part[b]; };

  // The attention kernels launched after this one may set themselves up now;
  // they read nothing of the plan (nor the cache) before the plan grid has completed.
  grid_dep_launch();
  // The lines of this thread's sequence lengths and of the start of its block
  // table row go into L2 while the previous grid finishes (prefetches read no
  // value: the loads below see any write the previous grid made).
  if (blockIdx.x == 0 && threadIdx.x < B) {
    prefetch_l2(p.cu_q + threadIdx.x);
    prefetch_l2(p.seq_lens + threadIdx.x);
    if (p.block_table) prefetch_l2(p.block_table + static_cast<size_t>(threadIdx.x) * p.bt_stride);
  }
  // This grid is itself a dependent launch: it may have become resident while
  // the kernel before it (the previous call's attention, or any other) still
  // ran, and it reads and writes nothing before that grid has completed.
  grid_dep_wait();
  if (blockIdx.x > 0) {
    write_new_rows(p);
    return;
  }
  if (threadIdx.x == 0) {
    s_tiles[0] = s_tiles[1] = 0ull;
    s_carry[0] = s_carry[1] = s_carry[2] = s_carry[3] = 0;
    s_need_zero = 0;
    s_dec_units = s_dec_max = 0;
    s_load[0] = s_load[1] = 0;
  }
  for (int i = threadIdx.x; i < 2 * kHistBuckets; i += NT) (&hist[0][0])[i] = 0;
  __syncthreads();

  // ---- pass 1: lengths, KV prefix (contiguous cache), q tile prefix, total work
  unsigned long long my_tiles[2] = {0ull, 0ull};
  unsigned my_dec_units = 0, my_dec_max = 0;
  for (int base = 0; base < B; base += NT) {
    const int b = base + threadIdx.x;
    int q0 = 0, ql = 0, L = 0, nqt = 0;
    bool ok = false;
    if (b < B) {
      q0 = p.cu_q[b];
      const int q1 = p.cu_q[b + 1];
      L = p.seq_lens[b];
      ql = q1 - q0;
      ok = q0 >= 0 && q1 >= q0 && q1 <= p.total_q && ql <= p.max_q && L >= 0 && L <= p.max_kv;
      if (!ok) atomicOr(ws.hdr + kHdrErr, kErrBadInput);
      // rows to zero: a rejected sequence's, or a first q tile that sees no key
      if (!ok || (ql > 0 && (L == 0 || (p.causal && L - ql + min(ql, p.tokens_per_tile) <= 0))))
        s_need_zero = 1;
      if (ok) {
        nqt = cdiv(ql, p.tokens_per_tile);
        // (both slots updated with a select: a run-time index would put the
        // array in local memory)
        const unsigned long long w = seq_blocks(p, ql, L, nqt);
        const bool dec = is_decode(p, ql);
        my_tiles[0] += dec ? 0ull : w;
        my_tiles[1] += dec ? w : 0ull;
        if (dec) {
          ++my_dec_units;
          my_dec_max = max(my_dec_max, static_cast<unsigned>(qtile_kv_tiles(p, ql, L, 0)));
        }
      }
    }
    int kv_excl, qt_excl;
    const int2 tot = block_exclusive_scan2<NT>(b < B ? max(L, 0) : 0, nqt, &kv_excl, &qt_excl, warp_sums);
    if (b < B) {
      // contiguous cache: the sequence's rows must lie inside the K/V planes
      if (ok && !p.block_table &&
          static_cast<long long>(s_carry[0]) + kv_excl + L > static_cast<long long>(p.num_pages)) {
        ok = false;
        atomicOr(ws.hdr + kHdrErr, kErrBadInput);
        s_need_zero = 1;
      }
      const int4 si = make_int4(q0, ok ? ql : -1, L, s_carry[0] + kv_excl);
      ws.seq_info[b] = si;
      ws.seq_plan[b] = make_int4(s_carry[1] + qt_excl, nqt, 1, 0);
      if (b < kSmemSeqs) s_qt_prefix[b] = s_carry[1] + qt_excl;
      if (b < kCacheSeqs) s_seq[b] = make_int4(q0, si.y, L, 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      s_carry[0] += tot.x;
      s_carry[1] += tot.y;
    }
    __syncthreads();
  }
  // total work: a warp sum, then one shared-memory atomic per warp that has any
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    my_tiles[k] = warp_sum_u64(my_tiles[k]);
    if (lane == 0 && my_tiles[k] != 0)
      atomicAdd(&s_tiles[k], my_tiles[k] * static_cast<unsigned long long>(p.n_heads_kv));
  }
  my_dec_units = __reduce_add_sync(0xffffffffu, my_dec_units);
  my_dec_max = __reduce_max_sync(0xffffffffu, my_dec_max);
  if (lane == 0 && my_dec_units != 0) {
    atomicAdd(&s_dec_units, static_cast<int>(my_dec_units));
    atomicMax(&s_dec_max, static_cast<int>(my_dec_max));
  }

  // ---- pass 1b: every live block-table entry must name a pool page (a warp per
  // sequence, eight independent loads per lane in flight)
  if (p.block_table) {
    for (int b = warp; b < B; b += NT / 32) {
      const int4 sq = seq_at(b);
      if (sq.y < 0) continue;
      const int np = cdiv(sq.z, kPage);
      const int32_t* row = p.block_table + static_cast<size_t>(b) * p.bt_stride;
      bool bad = false;
      for (int s0 = 0; s0 < np; s0 += 256) {
        int pg[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int s = s0 + u * 32 + lane;
          pg[u] = s < np ? row[s] : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) bad |= pg[u] < 0 || pg[u] >= p.num_pages;
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) {
        ws.seq_info[b].y = -1;
        if (b < kCacheSeqs) s_seq[b].y = -1;
        atomicOr(ws.hdr + kHdrErr, kErrBadInput);
        s_need_zero = 1;
      }
    }
  }
  __syncthreads();
  const int total_qt = s_carry[1];
  // the two kernels run one after the other, each over all SMs: each list's
  // split size comes from its own work and target
  auto chunk_for = [&](int k, int target) {
    const unsigned long long want = static_cast<unsigned long long>(max(target, 1));
    return max(static_cast<int>((s_tiles[k] + want - 1) / want), max(p.min_chunk, 1));
  };
  int dec_target = p.target_items;
  const int P = max(p.ctas, 1);
  const int dec_min_split_tiles = max(1, cdiv(p.min_chunk, kDecBlockN / kPage));
  const long long dec_units = static_cast<long long>(s_dec_units) * p.n_heads_kv;
  // skewed: longest unit > 2.5 x the mean unit. s_tiles[1] counts 64-key blocks (two per
  // decode tile) over all decode units, so mean = s_tiles[1] / (2 units) and the test is
  // max * units * 2 > 2.5 * s_tiles[1], i.e. 4 * max * units > 5 * s_tiles[1]
  const bool skewed = 4ull * static_cast<unsigned long long>(s_dec_max) * static_cast<unsigned long long>(dec_units) >
                      5ull * s_tiles[1];
  if (skewed && s_dec_max > dec_min_split_tiles && dec_units <= static_cast<long long>(kBalanceUnitsPerCta) * P) {
    // ---- the decode list's target, per call: counting sorts of its item costs
    // under both candidates (hist[0] and hist[1], still zero), then the largest
    // CTA load of each under the decode kernel's alternating round robin
    const int cand[2] = {p.target_items, p.target_items + p.target_items / 4};
    const int ct0 = max(1, cdiv(chunk_for(1, cand[0]), kDecBlockN / kPage));
    const int ct1 = max(1, cdiv(chunk_for(1, cand[1]), kDecBlockN / kPage));
    for (int b = threadIdx.x; b < B; b += NT) {
      const int4 sq = seq_at(b);
      if (sq.y <= 0 || !is_decode(p, sq.y)) continue;
      const int tiles = qtile_kv_tiles(p, sq.y, sq.z, 0);
      if (tiles == 0) continue;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int ct = j ? ct1 : ct0;
        const int S = tiles >= 2 ? min(min(cdiv(tiles, ct), kMaxSplits), tiles) : 1;
        for (int q = 0; q < S; ++q)
          atomicAdd(&hist[j][min((q + 1) * tiles / S - q * tiles / S, kHistBuckets - 1)], p.n_heads_kv);
      }
    }
    __syncthreads();
    int n_items0, n_items1;
    {
      const int2 tot = scan_hist_desc<NT>(hist, warp_sums);
      n_items0 = tot.x;
      n_items1 = tot.y;
      __syncthreads();
    }
    for (int t0 = 0; t0 < 2 * P; t0 += NT) {
      const int t = t0 + threadIdx.x;
      int load = 0, j = 0;
      if (t < 2 * P) {
        j = t / P;
        const int c = t - j * P;
        const int* start = hist[j];
        const int n_j = j ? n_items1 : n_items0;
        for (int k = 0, pos = c; pos < n_j; pos = cta_item(++k, c, P)) {
          // the cost of item `pos`: the largest bucket whose items begin at or before it
          int lo = 0, hi = kHistBuckets - 1;
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (start[mid - 1] > pos) lo = mid; else hi = mid - 1;
          }
          load += lo + kItemCost;
        }
      }
      // (P threads per candidate: a warp may straddle the two; reduce per candidate)
      const int l0 = __reduce_max_sync(0xffffffffu, (t < 2 * P && j == 0) ? load : 0);
      const int l1 = __reduce_max_sync(0xffffffffu, (t < 2 * P && j == 1) ? load : 0);
      if (lane == 0) {
        if (l0) atomicMax(&s_load[0], l0);
        if (l1) atomicMax(&s_load[1], l1);
      }
    }
    __syncthreads();
    if (s_load[1] < s_load[0]) dec_target = cand[1];
    for (int i = threadIdx.x; i < 2 * kHistBuckets; i += NT) (&hist[0][0])[i] = 0;
  }
  // (every thread sizes the chunks itself: no barrier)
  const int chunk_pre = chunk_for(0, p.target_items), chunk_dec = chunk_for(1, dec_target);

  // ---- pass 2: splits of single-q-tile units, partial rows and unit slots
  for (int base = 0; base < B; base += NT) {
    const int b = base + threadIdx.x;
    int S = 1, rows = 0;
    if (b < B) {
      const int4 sq = seq_at(b);
      if (sq.y > 0 && sq.y <= p.tokens_per_tile) {  // one q tile
        const int tiles = qtile_kv_tiles(p, sq.y, sq.z, 0);
        const bool dec = is_decode(p, sq.y);
        const int per_tile_shift = (dec ? kDecBlockNShift : p.block_n_shift) - kPageShift;
        const int chunk_tiles = max(1, ((dec ? chunk_dec : chunk_pre) + (1 << per_tile_shift) - 1) >> per_tile_shift);
        if (tiles >= 2) S = min(min(cdiv(tiles, chunk_tiles), kMaxSplits), tiles);
        rows = sq.y * G;
      }
    }
    const int part_rows = S >= 2 ? p.n_heads_kv * S * rows : 0;
    const int units = S >= 2 ? p.n_heads_kv : 0;
    int part_excl, unit_excl;
    const int2 tot = block_exclusive_scan2<NT>(part_rows, units, &part_excl, &unit_excl, warp_sums);
    if (b < B) {
      // (z, w) of the sequence's plan, stored without reading back its (x, y)
      const int2 sp = make_int2(S, s_carry[3] + unit_excl);
      *reinterpret_cast<int2*>(&ws.seq_plan[b].z) = sp;
      ws.seq_part[b] = s_carry[2] + part_excl;
      if (b < kCacheSeqs) {
        s_seq[b].w = S;
        s_part[b] = s_carry[2] + part_excl;
      }
      // the finished-split counters of the unit's KV heads start at zero (a plan
      // with more units than the workspace holds is rejected below)
      if (S >= 2 && sp.y + p.n_heads_kv <= ws.max_units)
        for (int hk = 0; hk < p.n_heads_kv; ++hk) ws.unit_cnt[sp.y + hk] = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      s_carry[2] += tot.x;
      s_carry[3] += tot.y;
    }
    __syncthreads();
  }
  const int total_part_rows = s_carry[2];
  const int total_units = s_carry[3];
  const bool overflow = total_part_rows > ws.max_part_rows || total_units > ws.max_units;

  // global q tile -> (sequence, q tile): the last sequence whose first q tile is <= gq
  auto seq_of_qtile = [&](int gq) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      const int x = mid < kSmemSeqs ? s_qt_prefix[mid] : ws.seq_plan[mid].x;
      if (x <= gq) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  auto qtile_first = [&](int b) { return b < kSmemSeqs ? s_qt_prefix[b] : ws.seq_plan[b].x; };

  // q tile qt of a sequence with ql queries makes an item unless it is the odd
  // half of a CTA pair's two q tiles; the item's KV tiles are those of its last
  // q tile (the later of a pair, which sees at least as many keys)
  auto item_tiles = [&](int ql, int L, int qt) -> int {
    if (p.pair && !is_decode(p, ql)) {
      if (qt & 1) return 0;
      return qtile_kv_tiles(p, ql, L, min(qt + 1, cdiv(ql, p.tokens_per_tile) - 1));
    }
    return qtile_kv_tiles(p, ql, L, qt);
  };

  // ---- pass 3: histogram of item costs (KV tiles per item), one per kernel
  if (!overflow) {
    for (int gq = threadIdx.x; gq < total_qt; gq += NT) {
      const int b = seq_of_qtile(gq);
      const int4 sq = seq_at(b);
      if (sq.y <= 0) continue;
      const int tiles = item_tiles(sq.y, sq.z, gq - qtile_first(b));
      if (tiles == 0) continue;
      const int list = is_decode(p, sq.y) ? 1 : 0;
      for (int s = 0; s < sq.w; ++s) {
        // (s <= 64 and tiles < 2^16: 32-bit products)
        const int k0 = s * tiles / sq.w;
        const int k1 = (s + 1) * tiles / sq.w;
        atomicAdd(&hist[list][min(k1 - k0, kHistBuckets - 1)], p.n_heads_kv);
      }
    }
  }
  __syncthreads();
  // exclusive scan of each list from the most expensive bucket down
  {
    const int2 tot = scan_hist_desc<NT>(hist, warp_sums);
    if (threadIdx.x == 0) {
      s_list_items[0] = tot.x;
      s_list_items[1] = tot.y;
    }
    __syncthreads();
  }
  const bool item_overflow = s_list_items[0] > ws.max_items || s_list_items[1] > ws.max_items;
  const bool bad_plan = overflow || item_overflow;

  // ---- pass 4: emit items, longest first, one KV head after the other, so
  // that within a cost bucket of the prefill list the items of one KV head
  // come out together: the persistent CTAs, which take the list in rounds of
  // one item each, then work on few KV heads at a time, and those heads' K/V
  // stay in L2 while every q tile of the head reads them. The decode list,
  // whose units read each page once, keeps the KV heads of a unit together
  // instead (a page holds all heads' rows). Positions within a bucket are
  // taken by atomics, so each head gets a sweep of its own, with a barrier
  // between sweeps. A prefill list of at most P / 2 items runs in one round on
  // any prefill kernel (all its items at once), where the order within a
  // bucket does not matter: it is emitted like the decode list, in one sweep.
  if (!bad_plan) {
    const bool one_round = s_list_items[0] <= P / 2;
    const int sweeps = one_round ? 1 : p.n_heads_kv;
    for (int hk_t = 0; hk_t < sweeps; ++hk_t) {
      for (int gq = threadIdx.x; gq < total_qt; gq += NT) {
        const int b = seq_of_qtile(gq);
        const int4 sq = seq_at(b);
        if (sq.y <= 0) continue;
        const int list = is_decode(p, sq.y) ? 1 : 0;
        const bool all_heads = list == 1 || one_round;  // the unit's heads together, in one sweep
        const int qt = gq - qtile_first(b);
        const int tiles = item_tiles(sq.y, sq.z, qt);
        if (tiles == 0) continue;
        const int S = sq.w;
        const int rows = sq.y * G;
        const int nh = all_heads ? p.n_heads_kv : 1;
        if (all_heads && hk_t != 0) continue;  // (emitted by the sweep of head 0)
        int4* dst = list ? ws.dec_items : ws.items;
        const int part0 = S >= 2 ? part_at(b) : 0;
        for (int s = 0; s < S; ++s) {
          const int k0 = s * tiles / S;
          const int k1 = (s + 1) * tiles / S;
          const int pos = atomicAdd(&hist[list][min(k1 - k0, kHistBuckets - 1)], nh);
          for (int j = 0; j < nh; ++j) {
            const int hk = hk_t + j;
            if (S >= 2)  // split s of the (b, hk) unit (q tile 0)
              dst[pos + j] = make_int4(b | (s << kSeqBits), hk << 16, (k0 << 16) | k1,
                                       part0 + (hk * S + s) * rows);
            else
              dst[pos + j] = make_int4(b, (hk << 16) | qt, (k0 << 16) | k1, -1);
          }
        }
      }
      __syncthreads();
    }
  }

  // ---- zero fill: rejected sequences and q tiles that see no key (all rows of
  // every sequence if the workspace could not hold the plan). Each thread takes
  // whole sequences; only degenerate inputs reach the stores, and the walk is
  // skipped when pass 1 saw none.
  for (int b = threadIdx.x; (s_need_zero || bad_plan) && b < B; b += NT) {
    // the query range of a live sequence from the cached plan; a rejected one's
    // from cu_q (it may be out of range)
    const int4 sq = seq_at(b);
    int q0 = sq.x, q1 = sq.x + sq.y;
    if (sq.y < 0) {
      q0 = p.cu_q[b];
      q1 = p.cu_q[b + 1];
    }
    if (!(q0 >= 0 && q1 >= q0 && q1 <= p.total_q) || q1 == q0) continue;
    int z1 = q0;  // rows [q0, z1) get zeros
    if (sq.y < 0 || bad_plan) {
      z1 = q1;
    } else {
      const int nqt = cdiv(sq.y, p.tokens_per_tile);
      for (int qt = 0; qt < nqt && qtile_kv_tiles(p, sq.y, sq.z, qt) == 0; ++qt)
        z1 = q0 + min(sq.y, (qt + 1) * p.tokens_per_tile);
    }
    if (z1 > q0 && p.out) {  // (no output when only the quantised Q/K are wanted)
      const size_t row = static_cast<size_t>(p.n_heads_q) * p.head_dim;
      uint4* o = reinterpret_cast<uint4*>(p.out + static_cast<size_t>(q0) * row);
      const size_t n16 = static_cast<size_t>(z1 - q0) * row / 8;
      for (size_t i = 0; i < n16; ++i) o[i] = make_uint4(0, 0, 0, 0);
    }
  }
  if (threadIdx.x == 0) {
    ws.hdr[kHdrItems] = bad_plan ? 0 : s_list_items[0];
    ws.hdr[kHdrDecItems] = bad_plan ? 0 : s_list_items[1];
    ws.hdr[kHdrUnits] = bad_plan ? 0 : total_units;
    ws.hdr[kHdrPartRows] = total_part_rows;
    ws.hdr[kHdrOverflow] = bad_plan ? 1 : 0;
    ws.hdr[kHdrGo] = 0;  // set by the decode kernel once this grid has completed
    if (bad_plan) atomicOr(ws.hdr + kHdrErr, kErrBadInput);
  }
}

// A bounded wait that nothing ends: one warp waits on a fresh mbarrier for a
// phase no thread completes, with the attention kernels' own wait helper, so
// that after its time limit it sets the abort flag and the timeout bit of the
// device error word and returns (the self-test of failure detection).
__global__ void __launch_bounds__(32) wait_selftest_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_addr(&bar), 1);
    mbar_init_fence();
  }
  __syncwarp();
  const WaitCtl ctl{&abort_flag, err};
  wait_warp(smem_addr(&bar), 0, ctl);
}

}  // namespace


cudaError_t launch_plan(const PlanParams& p, cudaStream_t s, bool dependent) {
  // small batches: at most 32 sequences (the block-table check, a warp per
  // sequence, then takes at most 8 rounds of its four warps) and 256 q tiles
  const long long qtiles_bound =
      (static_cast<long long>(p.total_q) + p.tokens_per_tile - 1) / std::max(p.tokens_per_tile, 1) + p.num_seqs;
  if (p.num_seqs <= kPlanSmallSeqs && qtiles_bound <= 2 * kPlanThreadsSmall) {
    // the cache-write CTAs keep a warp per 32 tokens at most, as with the large CTA
    constexpr int kWarpsSmall = kPlanThreadsSmall / 32;
    const int write =
        p.write_ctas > 0 ? std::min((p.total_q + kWarpsSmall - 1) / kWarpsSmall, 8 * p.write_ctas) : 0;
    return launch_kernel(plan_kernel<kPlanThreadsSmall>, dim3(1 + write), dim3(kPlanThreadsSmall), 0, s,
                         dependent, p);
  }
  return launch_kernel(plan_kernel<kPlanThreads>, dim3(1 + p.write_ctas), dim3(kPlanThreads), 0, s, dependent, p);
}

cudaError_t launch_wait_selftest(int* err, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(err);
  return cudaGetLastError();
}

}  // namespace pattn
