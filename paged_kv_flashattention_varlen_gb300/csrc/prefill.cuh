// prefill.cuh -- pieces shared by the prefill attention kernels (attn.cu, the
// one-q-tile kernels; attn2q.cu, the two-q-tile kernel): the work item of the
// planned list and the end of a split item (count it in its unit; the CTA that
// finishes the unit's last split merges the unit).
#pragma once
#include "kernels.cuh"
#include "merge.cuh"
#include "ptx.cuh"

namespace pattn {

constexpr int kSoftmaxWarps = 8;  // warps 4-11 of a prefill CTA

// The start of a prefill CTA: the plan grid must be complete. With
// p.early_start that is the go word (set by the decode kernel past its own
// grid wait: thread 0 waits for it, bounded; then every thread reads it with
// acquire ordering), else the grid before this one. Returns false when the
// wait ran out (the abort flag and the timeout bit are set).
__device__ __forceinline__ bool prefill_start(const AttnParams& p, const WaitCtl& ctl) {
  if (!p.early_start) {
    grid_dep_wait();
    return true;
  }
  if (threadIdx.x == 0) {
    const uint64_t t0 = global_ns();
    for (uint32_t n = 0; ld_acquire_gpu(p.go) == 0; ++n) {
      if ((n & 15u) == 15u && global_ns() - t0 > kWaitLimitNs) {
        *ctl.abort = 1;
        atomicOr(ctl.err, kErrTimeout);
        break;
      }
      __nanosleep(100);
    }
  }
  __syncthreads();
  (void)ld_acquire_gpu(p.go);
  return *ctl.abort == 0;
}

// The end of a prefill CTA: with p.early_start, wait for the grid before
// this one (the decode kernel), so that this grid completes after it.
__device__ __forceinline__ void prefill_end(const AttnParams& p) {
  if (p.early_start) grid_dep_wait();
}

// part: first partial row of this split, -1 if the item is not split; split:
// the split's index in its unit.
struct Item {
  int b, hk, qt, kt0, kt1, part, split;
};

__device__ __forceinline__ Item decode_item(int4 v) {
  Item it;
  it.b = v.x & kSeqMask;
  it.hk = v.y >> 16;
  it.qt = v.y & 0xFFFF;
  it.kt0 = (v.z >> 16) & 0xFFFF;
  it.kt1 = v.z & 0xFFFF;
  it.part = v.w;
  it.split = v.x >> kSeqBits;
  return it;
}

// After a split item's partials are written (softmax warps 4-11): count the
// split in its unit's counter; the CTA that finishes the unit's last split
// merges the unit's rows (the decode manifest's last-CTA reduction through its
// counter scratch). Bounded waits only: warp 4 takes the count once all eight
// warps have fenced their writes, then releases them with the result.
template <int D>
__device__ __forceinline__ bool split_done(const AttnParams& p, const Item& it, int4 si, uint32_t bar_a,
                                           uint32_t bar_b, volatile int* flag, uint32_t& nsp, int warp,
                                           const WaitCtl& ctl) {
  const int lane = threadIdx.x & 31;
  __threadfence();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar_a);
  bool ok = true;
  if (warp == 4) {
    if (lane == 0) {
      ok = wait_one(bar_a, nsp & 1u, ctl);
      int last = 0;
      if (ok) {
        const int4 sp = p.seq_plan[it.b];
        last = atomicAdd(&p.unit_cnt[sp.w + it.hk], 1) == sp.z - 1;
        if (last) __threadfence();
      }
      *flag = last;
      mbar_arrive(bar_b);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
  }
  if (!wait_warp(bar_b, nsp & 1u, ctl)) ok = false;
  ++nsp;
  if (!ok) return false;
  if (*flag) {
    const int4 sp = p.seq_plan[it.b];
    const int rows = si.y * p.group;
    merge_unit<D, 1>(p, si.x, it.hk, sp.z, it.part - it.split * rows, rows, warp - 4, kSoftmaxWarps);
  }
  return true;
}

}  // namespace pattn
