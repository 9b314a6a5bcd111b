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
//   3. splits the KV range of single-q-tile units (decode) so that the whole
//      job has about `target_items` items of at least `min_chunk` tiles (the
//      decode manifest's "MultiCtasKv": several CTAs per sequence and KV
//      head, with partial O and (max, sum) statistics in scratch);
//   4. orders the items longest first (counting sort on the number of KV
//      tiles) so that round-robin assignment to persistent CTAs balances;
//   5. zero-fills the output rows of q tiles that see no key at all, and
//      zeroes the finished-split counter of every split unit (the decode
//      kernel merges a unit's partials in the CTA that finishes it last).
//
// merge_kernel merges the split units of the prefill kernel's items (one per
// unit, found at its split-0 item), after that kernel.
#include "kernels.cuh"
#include "merge.cuh"
#include "ptx.cuh"

namespace pattn {
namespace {

constexpr int kPlanThreads = 1024;

// Block-wide exclusive scan of one int per thread; returns the block total.
__device__ int block_exclusive_scan(int v, int* out_excl, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const int before = warp ? warp_sums[warp - 1] : 0;
  *out_excl = before + x - v;
  const int total = warp_sums[31];
  __syncthreads();
  return total;
}

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Units of at most kDecRows packed rows run on the swap-AB decode kernel.
__device__ __forceinline__ bool is_decode(const PlanParams& p, int ql) {
  return p.dec_enabled && ql >= 1 && ql * p.group <= kDecRows;
}

// Visible KV tiles of q tile qt: keys [0, kv_hi), kv_hi the largest limit of its rows.
__device__ __forceinline__ int qtile_kv_tiles(const PlanParams& p, int ql, int L, int qt) {
  int hi = L;
  if (p.causal) {
    const int last_tok = min(ql, (qt + 1) * p.tokens_per_tile);
    hi = min(L, L - ql + last_tok);
  }
  const int bn = is_decode(p, ql) ? kDecBlockN : p.block_n;
  return hi > 0 ? cdiv(hi, bn) : 0;
}

// Work of a q tile in 64-key blocks (comparable across the two kernels' tile sizes).
__device__ __forceinline__ int qtile_blocks(const PlanParams& p, int ql, int L, int qt) {
  const int bn = is_decode(p, ql) ? kDecBlockN : p.block_n;
  return qtile_kv_tiles(p, ql, L, qt) * (bn / kPage);
}

constexpr int kSmemSeqs = 4096;  // sequences whose q-tile prefix is kept in shared memory

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(const PlanParams p) {
  __shared__ int warp_sums[32];
  __shared__ int hist[2][kHistBuckets];  // [0] prefill items, [1] decode items
  __shared__ int s_qt_prefix[kSmemSeqs];
  __shared__ int s_carry[4];
  __shared__ unsigned long long s_tiles;
  __shared__ int s_chunk;
  __shared__ int s_total_items;
  const Workspace& ws = p.ws;
  const int B = p.num_seqs;
  const int G = p.group;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    s_tiles = 0ull;
    s_carry[0] = s_carry[1] = s_carry[2] = s_carry[3] = 0;
  }
  __syncthreads();

  // ---- pass 1: lengths, KV prefix (contiguous cache), q tile prefix, total tiles
  unsigned long long my_tiles = 0;
  for (int base = 0; base < B; base += kPlanThreads) {
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
      if (ok) {
        nqt = cdiv(ql, p.tokens_per_tile);
        for (int qt = 0; qt < nqt; ++qt)
          my_tiles += static_cast<unsigned long long>(qtile_blocks(p, ql, L, qt));
      }
    }
    int kv_excl, qt_excl;
    const int kv_tot = block_exclusive_scan(b < B ? max(L, 0) : 0, &kv_excl, warp_sums);
    const int qt_tot = block_exclusive_scan(nqt, &qt_excl, warp_sums);
    if (b < B) {
      // contiguous cache: the sequence's rows must lie inside the K/V planes
      if (ok && !p.block_table &&
          static_cast<long long>(s_carry[0]) + kv_excl + L > static_cast<long long>(p.num_pages)) {
        ok = false;
        atomicOr(ws.hdr + kHdrErr, kErrBadInput);
      }
      ws.seq_info[b] = make_int4(q0, ok ? ql : -1, L, s_carry[0] + kv_excl);
      ws.seq_plan[b] = make_int4(s_carry[1] + qt_excl, nqt, 1, 0);
      if (b < kSmemSeqs) s_qt_prefix[b] = s_carry[1] + qt_excl;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      s_carry[0] += kv_tot;
      s_carry[1] += qt_tot;
    }
    __syncthreads();
  }
  atomicAdd(&s_tiles, my_tiles * static_cast<unsigned long long>(p.n_heads_kv));

  // ---- pass 1b: every live block-table entry must name a pool page (warp per sequence)
  if (p.block_table) {
    for (int b = warp; b < B; b += kPlanThreads / 32) {
      const int4 si = ws.seq_info[b];
      if (si.y < 0) continue;
      const int np = cdiv(si.z, kPage);
      bool bad = false;
      for (int s = lane; s < np; s += 32) {
        const int pg = p.block_table[static_cast<size_t>(b) * p.bt_stride + s];
        bad |= pg < 0 || pg >= p.num_pages;
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) {
        ws.seq_info[b].y = -1;
        atomicOr(ws.hdr + kHdrErr, kErrBadInput);
      }
    }
  }
  __syncthreads();
  const int total_qt = s_carry[1];
  if (threadIdx.x == 0) {
    const unsigned long long t = s_tiles;
    const unsigned long long want = static_cast<unsigned long long>(max(p.target_items, 1));
    const int chunk = static_cast<int>((t + want - 1) / want);
    s_chunk = max(chunk, max(p.min_chunk, 1));
    s_carry[2] = s_carry[3] = 0;
  }
  __syncthreads();
  const int chunk = s_chunk;

  // ---- pass 2: splits of single-q-tile units, partial rows and unit slots
  for (int base = 0; base < B; base += kPlanThreads) {
    const int b = base + threadIdx.x;
    int S = 1, rows = 0;
    if (b < B) {
      const int4 si = ws.seq_info[b];
      const int nqt = ws.seq_plan[b].y;
      if (si.y > 0 && nqt == 1) {
        const int tiles = qtile_kv_tiles(p, si.y, si.z, 0);
        const int per_tile = qtile_blocks(p, si.y, si.z, 0) / max(tiles, 1);  // 64-key blocks
        const int chunk_tiles = max(1, cdiv(chunk, max(per_tile, 1)));
        if (tiles >= 2) S = min(min(cdiv(tiles, chunk_tiles), kMaxSplits), tiles);
        rows = si.y * G;
      }
    }
    const int part_rows = S >= 2 ? p.n_heads_kv * S * rows : 0;
    const int units = S >= 2 ? p.n_heads_kv : 0;
    int part_excl, unit_excl;
    const int part_tot = block_exclusive_scan(part_rows, &part_excl, warp_sums);
    const int unit_tot = block_exclusive_scan(units, &unit_excl, warp_sums);
    if (b < B) {
      int4 sp = ws.seq_plan[b];
      sp.z = S;
      sp.w = s_carry[3] + unit_excl;
      ws.seq_plan[b] = sp;
      ws.seq_part[b] = s_carry[2] + part_excl;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      s_carry[2] += part_tot;
      s_carry[3] += unit_tot;
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

  // ---- pass 3: histogram of item costs (KV tiles per item), one per kernel
  for (int i = threadIdx.x; i < 2 * kHistBuckets; i += kPlanThreads) (&hist[0][0])[i] = 0;
  __syncthreads();
  if (!overflow) {
    for (int gq = threadIdx.x; gq < total_qt; gq += kPlanThreads) {
      const int b = seq_of_qtile(gq);
      const int4 sp = ws.seq_plan[b];
      const int4 si = ws.seq_info[b];
      if (si.y <= 0) continue;
      const int tiles = qtile_kv_tiles(p, si.y, si.z, gq - sp.x);
      if (tiles == 0) continue;
      const int list = is_decode(p, si.y) ? 1 : 0;
      for (int s = 0; s < sp.z; ++s) {
        const int k0 = static_cast<int>(static_cast<long long>(s) * tiles / sp.z);
        const int k1 = static_cast<int>(static_cast<long long>(s + 1) * tiles / sp.z);
        atomicAdd(&hist[list][min(k1 - k0, kHistBuckets - 1)], p.n_heads_kv);
      }
    }
  }
  __syncthreads();
  // exclusive scan of each list from the most expensive bucket down
  __shared__ int s_list_items[2];
  for (int list = 0; list < 2; ++list) {
    constexpr int kPer = kHistBuckets / kPlanThreads;
    int local[kPer];
    int sum = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      local[k] = hist[list][kHistBuckets - 1 - (threadIdx.x * kPer + k)];
      sum += local[k];
    }
    int excl;
    const int tot = block_exclusive_scan(sum, &excl, warp_sums);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      hist[list][kHistBuckets - 1 - (threadIdx.x * kPer + k)] = excl;
      excl += local[k];
    }
    if (threadIdx.x == 0) s_list_items[list] = tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) s_total_items = max(s_list_items[0], s_list_items[1]);
  __syncthreads();
  const bool item_overflow = s_total_items > ws.max_items;
  const bool bad_plan = overflow || item_overflow;

  // ---- pass 4: emit items, longest first
  if (!bad_plan) {
    for (int gq = threadIdx.x; gq < total_qt; gq += kPlanThreads) {
      const int b = seq_of_qtile(gq);
      const int4 sp = ws.seq_plan[b];
      const int4 si = ws.seq_info[b];
      if (si.y <= 0) continue;
      const int qt = gq - sp.x;
      const int tiles = qtile_kv_tiles(p, si.y, si.z, qt);
      if (tiles == 0) continue;
      const int S = sp.z;
      const int rows = si.y * G;
      const int list = is_decode(p, si.y) ? 1 : 0;
      int4* dst = list ? ws.dec_items : ws.items;
      for (int s = 0; s < S; ++s) {
        const int k0 = static_cast<int>(static_cast<long long>(s) * tiles / S);
        const int k1 = static_cast<int>(static_cast<long long>(s + 1) * tiles / S);
        const int pos = atomicAdd(&hist[list][min(k1 - k0, kHistBuckets - 1)], p.n_heads_kv);
        for (int hk = 0; hk < p.n_heads_kv; ++hk) {
          if (S >= 2)  // split s of the (b, hk) unit (q tile 0)
            dst[pos + hk] = make_int4(b | (s << kSeqBits), hk << 16, (k0 << 16) | k1,
                                      ws.seq_part[b] + (hk * S + s) * rows);
          else
            dst[pos + hk] = make_int4(b, (hk << 16) | qt, (k0 << 16) | k1, -1);
        }
      }
    }
    // finished-split counters of the split units start at zero
    for (int b = threadIdx.x; b < B; b += kPlanThreads) {
      const int4 sp = ws.seq_plan[b];
      if (sp.z < 2) continue;
      for (int hk = 0; hk < p.n_heads_kv; ++hk) ws.unit_cnt[sp.w + hk] = 0;
    }
  }

  // ---- zero fill: rejected sequences and q tiles that see no key (all rows of
  // every sequence if the workspace could not hold the plan). Each thread takes
  // whole sequences; only degenerate inputs reach the stores.
  for (int b = threadIdx.x; b < B; b += kPlanThreads) {
    const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
    if (!(q0 >= 0 && q1 >= q0 && q1 <= p.total_q) || q1 == q0) continue;
    const int4 si = ws.seq_info[b];
    int z1 = q0;  // rows [q0, z1) get zeros
    if (si.y < 0 || bad_plan) {
      z1 = q1;
    } else {
      const int nqt = ws.seq_plan[b].y;
      for (int qt = 0; qt < nqt && qtile_kv_tiles(p, si.y, si.z, qt) == 0; ++qt)
        z1 = q0 + min(si.y, (qt + 1) * p.tokens_per_tile);
    }
    if (z1 > q0) {
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
    if (bad_plan) atomicOr(ws.hdr + kHdrErr, kErrBadInput);
  }
}

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const AttnParams p) {
  const int n_items = p.hdr[kHdrItems];
  const int warp = threadIdx.x >> 5;
  for (int idx = blockIdx.x; idx < n_items; idx += gridDim.x) {
    const int4 iv = p.items[idx];
    if (iv.w < 0 || (iv.x >> kSeqBits) != 0) continue;  // one CTA per unit: its split 0
    const int b = iv.x & kSeqMask;
    const int4 si = p.seq_info[b];
    const int4 sp = p.seq_plan[b];
    merge_unit<D>(p, si.x, iv.y >> 16, sp.z, iv.w, si.y * p.group, warp, 8);
  }
}

}  // namespace

cudaError_t launch_merge(const AttnParams& p, int head_dim, int grid, cudaStream_t s) {
  if (head_dim == 128)
    merge_kernel<128><<<grid, 256, 0, s>>>(p);
  else
    merge_kernel<256><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t s) {
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pattn
