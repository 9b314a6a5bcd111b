// kvwrite.cu -- the cache write in front of attention: the K and V rows of the
// new tokens go into their slots of the paged (or contiguous) KV cache, the
// `reshape_and_cache_flash` node that comes right before `attend` in the GB10
// model graph (P4, "kv_write", state "k:write,v:write", steps "cache bf16").
//
// Token i of sequence b (i < ql_b) is cache position L_b - ql_b + i, the same
// bottom-right alignment the attention uses: slot (pos / page_size) of the
// block table and row pos % page_size of that page; in a contiguous cache,
// row pos of the sequence. The kernel runs after the plan kernel (it reads the
// plan's validated lengths and contiguous row offsets, and writes nothing for
// a sequence the plan rejected) and before the attention kernels, all on one
// stream; it is a dependent launch, so its CTAs are resident while the plan
// finishes, and the attention kernels' device-side wait covers it.
//
// HBM-bound copy: one warp per token, 16-byte loads and stores of the token's
// contiguous K row and V row ([Hkv][D] each) with all loads of a row issued
// before its stores.
#include "kernels.cuh"
#include "ptx.cuh"

namespace pattn {
namespace {

constexpr int kKvwThreads = 256;

__global__ void __launch_bounds__(kKvwThreads) kv_write_kernel(const KvWriteParams p) {
  grid_dep_launch();  // the attention kernels may set themselves up now
  grid_dep_wait();    // the plan is complete: seq_info holds validated lengths
  const int lane = threadIdx.x & 31;
  const int warps = static_cast<int>(gridDim.x) * (kKvwThreads / 32);
  const int w = static_cast<int>(blockIdx.x) * (kKvwThreads / 32) + (threadIdx.x >> 5);
  // tokens [t0, t1) of this warp, walked in order so that the sequence index
  // only moves forward
  const int per = (p.total_q + warps - 1) / warps;
  const int t0 = w * per, t1 = min(p.total_q, t0 + per);
  if (t0 >= t1) return;
  // sequence of token t0: the last b with cu_q[b] <= t0
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu_q[mid] <= t0) lo = mid; else hi = mid - 1;
  }
  int b = lo;
  const int n16 = p.row_elems / 8;  // 16-byte chunks of one token's K (or V) row
  for (int t = t0; t < t1; ++t) {
    while (b + 1 < p.num_seqs && p.cu_q[b + 1] <= t) ++b;
    const int4 si = p.seq_info[b];
    if (si.y < 0) continue;  // rejected by the plan: its rows were zero-filled
    const int pos = si.z - si.y + (t - si.x);
    if (pos < 0) continue;   // more queries than keys: no slot for this token
    size_t krow, vrow;       // element offsets of the destination rows
    if (p.block_table) {
      const int page = p.block_table[static_cast<size_t>(b) * p.bt_stride + pos / kPage];
      if (page < 0 || page >= p.num_pages) {
        if (lane == 0) atomicOr(p.err, kErrBadInput);
        continue;
      }
      krow = (static_cast<size_t>(page) * 2 * kPage + (pos % kPage)) * p.row_elems;
      vrow = krow + static_cast<size_t>(kPage) * p.row_elems;
    } else {
      krow = (static_cast<size_t>(si.w) + pos) * p.row_elems;
      vrow = krow + static_cast<size_t>(p.num_pages) * p.row_elems;
    }
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_new + static_cast<size_t>(t) * p.row_elems);
    const uint4* vs = reinterpret_cast<const uint4*>(p.v_new + static_cast<size_t>(t) * p.row_elems);
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

}  // namespace

cudaError_t launch_kv_write(const KvWriteParams& p, int sms, cudaStream_t s) {
  const int warps_needed = p.total_q;
  const int blocks = std::max(1, std::min((warps_needed + kKvwThreads / 32 - 1) / (kKvwThreads / 32), 4 * sms));
  return launch_kernel(kv_write_kernel, blocks, kKvwThreads, 0, s, true, p);
}

}  // namespace pattn
