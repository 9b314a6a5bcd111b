// kernels.cuh -- parameters shared by the host side and the device kernels
// (plan, cache write, quantisation, decode and prefill attention) of the
// paged-KV varlen attention library.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

namespace pattn {

constexpr int kBM = 128;            // packed query rows per tile (tokens x GQA group)
constexpr int kPage = 64;           // page size handled by the gather (rows per TMA box)
constexpr int kThreads = 288;       // decode kernel: load, QK MMA, V tail fix, split merge, 4 x softmax, PV MMA
constexpr int kTmemCols = 512;
constexpr int kHistBuckets = 1024;  // cost buckets of the longest-first order, per item list
constexpr int kDecRows = 16;        // packed query rows a swap-AB decode item holds
constexpr int kDecBlockN = 128;     // keys per KV tile of the decode kernel
constexpr int kDecBlockNShift = 7;
constexpr int kPageShift = 6;
static_assert(kDecBlockN == 1 << kDecBlockNShift && kPage == 1 << kPageShift, "tile shifts");
constexpr int kMaxSplits = 64;

// Bits of the device error word.
constexpr int kErrBadInput = 1;
constexpr int kErrTimeout = 2;

// Device workspace header (int words).
// kHdrGo: the plan grid has completed (reset by the plan, set by the decode
// kernel's first CTA once past its own grid wait); see AttnParams::early_start.
enum HdrWord { kHdrErr = 0, kHdrItems = 1, kHdrUnits = 2, kHdrPartRows = 3, kHdrOverflow = 4,
               kHdrDecItems = 5, kHdrGo = 6, kHdrWords = 64 };

// Work item, 16 bytes:
//   x = sequence b (bits 0-23) | split index << 24 (split items)
//   y = kv head << 16 | q tile (0 for split items: their unit has one q tile)
//   z = first kv tile << 16 | end kv tile
//   w = -1: not split, the item writes bf16 out directly;
//       >= 0: first partial row of this split (split s of a unit with `rows`
//       packed rows; the unit's partials start at w - s * rows)
constexpr int kSeqBits = 24;
constexpr int kSeqMask = (1 << kSeqBits) - 1;
// Sequence info, 16 bytes: x = first query token, y = query length (-1: rejected),
//   z = KV length, w = first KV row (contiguous cache).

struct Workspace {
  int* hdr;
  int4* seq_info;
  int4* seq_plan;   // x = first global q tile, y = q tiles, z = splits, w = first split unit
  int* unit_cnt;    // finished splits per split unit (zeroed by the plan)
  int* seq_part;    // first partial row of the sequence's split units
  int4* items;      // prefill kernel items
  int4* dec_items;  // swap-AB decode kernel items
  float* part_o;    // [rows][D] split-normalised partial O
  float2* part_ml;  // [rows] (running max in log2 units, sum of exp2)
  int max_items;
  int max_units;
  int max_part_rows;
};

struct PlanParams {
  const int32_t* cu_q;
  const int32_t* seq_lens;
  const int32_t* block_table;  // nullptr: contiguous cache
  __nv_bfloat16* out;
  Workspace ws;
  int num_seqs, total_q, max_q, max_kv;
  int n_heads_q, n_heads_kv, group, head_dim;
  int tokens_per_tile;  // T = kBM / group
  int block_n;          // keys per KV tile of the prefill kernel
  int block_n_shift;    // log2(block_n)
  int pair;             // prefill items of two q tiles (CTA-pair kernel, two-q-tile kernel)
  int dec_enabled;      // group <= kDecRows: units of <= kDecRows packed rows go to the decode kernel
  int bt_stride, num_pages;
  int causal;
  int target_items;     // items per list the split heuristic aims at (a multiple of the SM count);
                        // the decode list may take target_items + target_items / 4 instead
  int min_chunk;        // fewest KV tiles per split
  int ctas;             // persistent CTAs of the decode kernel (its grid)
  // cache write of the new tokens (pattn_forward_append): CTAs 1..write_ctas of
  // the plan grid copy k_new / v_new [total_q][n_heads_kv][head_dim] into the
  // pool while CTA 0 plans; write_ctas = 0 and null pointers otherwise
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  __nv_bfloat16* kv_pool;
  int write_ctas;
};

// Preparation of the quantised variants (quant.cu). Layouts:
//   q8 [total_q][n_heads_q][head_dim] e4m3, q_scale [total_q][n_heads_q] fp32;
//   k8 [num_seqs * nb_max][64][n_heads_kv][head_dim] e4m3 (sequence b's 64-key
//   block j is block b * nb_max + j), k_scale [num_seqs * nb_max][n_heads_kv];
//   v8 [num_seqs * nb_max / 2][n_heads_kv][head_dim][128] e4m3: V transposed,
//   keys innermost, 128-key tile t of sequence b at b * nb_max / 2 + t, zero
//   codes past the sequence end; v_scale [num_seqs][n_heads_kv][head_dim] fp32.
//   Scratch (quant_scratch_bytes), per (sequence, KV head): first, zeroed before
//   the call (quant_zero_bytes), k_sum [..][head_dim] int64 (units of 2^-32),
//   v_amax [..][head_dim] uint32 (fp32 bits of max |v|), k_cnt [..] uint32;
//   then k_mean [..][head_dim] fp32 and v_inv [..][head_dim] fp32 (448 / amax).
struct QuantScratch {
  long long* k_sum;
  unsigned int* v_amax;
  unsigned int* k_cnt;
  float* k_mean;
  float* v_inv;
};
inline size_t quant_zero_bytes(int num_seqs, int n_heads_kv, int head_dim) {
  const size_t n = static_cast<size_t>(num_seqs) * n_heads_kv;
  return n * head_dim * (sizeof(long long) + sizeof(unsigned int)) + n * sizeof(unsigned int);
}
inline size_t quant_scratch_bytes(int num_seqs, int n_heads_kv, int head_dim) {
  const size_t n = static_cast<size_t>(num_seqs) * n_heads_kv;
  return (quant_zero_bytes(num_seqs, n_heads_kv, head_dim) + 15) / 16 * 16 + 2 * n * head_dim * sizeof(float);
}
inline QuantScratch quant_scratch_split(void* base, int num_seqs, int n_heads_kv, int head_dim) {
  const size_t n = static_cast<size_t>(num_seqs) * n_heads_kv, nd = n * head_dim;
  uint8_t* b = static_cast<uint8_t*>(base);
  QuantScratch q;
  q.k_sum = reinterpret_cast<long long*>(b);
  q.v_amax = reinterpret_cast<unsigned int*>(b + nd * sizeof(long long));
  q.k_cnt = q.v_amax + nd;
  q.k_mean = reinterpret_cast<float*>(b + (quant_zero_bytes(num_seqs, n_heads_kv, head_dim) + 15) / 16 * 16);
  q.v_inv = q.k_mean + nd;
  return q;
}

struct QuantParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kv_pool;
  const int32_t* block_table;
  const int4* seq_info;
  uint8_t* q8;       // nullptr: no Q codes
  float* q_scale;
  uint8_t* k8;       // nullptr: no K codes
  float* k_scale;
  uint8_t* v8;       // nullptr: no V codes (nor V maxima)
  float* v_scale;
  QuantScratch sc;
  int num_seqs, total_q, n_heads_q, n_heads_kv, head_dim, bt_stride, num_pages;
  int nb_max;  // 64-key blocks per sequence in k8 (even): 2 * ceil(max_kv / 128)
};

struct AttnParams {
  const int4* items;
  const int* hdr;
  const int4* seq_info;
  const int32_t* block_table;
  __nv_bfloat16* out;
  float* part_o;
  float2* part_ml;
  int* err;
  int bt_stride, num_pages;
  int n_heads_q, n_heads_kv, group, tokens_per_tile;
  float scale_log2;  // softmax scale * log2(e)
  int causal;
  int paged;
  const int4* seq_plan;  // z = splits, w = first split unit of the sequence
  int* unit_cnt;         // finished splits per split unit
  // quantised-QK variant: e4m3 scales of Q rows [total_q][n_heads_q] and of K
  // blocks [num_seqs * nb_max][n_heads_kv] (see QuantParams)
  const float* q_scale;
  const float* k_scale;
  int nb_max;
  // fp8 P.V variant: per-channel V scales [num_seqs][n_heads_kv][head_dim]
  const float* v_scale;
  // failure-detection self-test only (0 otherwise): the first CTA's MMA-issuing
  // thread waits for a barrier phase that nothing completes, so that its
  // bounded wait runs out and the CTA takes its abort-and-drain path
  int selftest_abort;
  // the workspace's kHdrGo word: the decode kernel sets it once past its grid
  // wait. With early_start (both attention kernels launched), the prefill kernel
  // starts on it rather than on the decode grid, so that its CTAs work as soon
  // as they hold an SM (the decode kernel's last CTAs may still run); each of
  // its CTAs waits for the decode grid before it exits, so the prefill grid
  // still completes after it, as stream order requires.
  int* go;
  int early_start;
};


// Launchers (defined in the .cu files; return the launch error).
// The k-th work item of CTA c out of P. The item lists are sorted longest first
// and the rounds alternate direction (c, 2P-1-c, 2P+c, 4P-1-c, ...), so that
// each CTA's share of the sorted costs comes out about even. Increasing in k.
__device__ __forceinline__ int cta_item(int k, int c, int P) {
  return (k & 1) ? (k + 1) * P - 1 - c : k * P + c;
}

// Kernel launch; with `dependent` the grid may begin (up to its grid_dep_wait)
// while the previous grid in the stream finishes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, bool dependent, const Args&... args) {
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = &attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The same for a kernel whose CTAs run as pairs (clusters of two).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel_pair(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t s, bool dependent, const Args&... args) {
  cudaLaunchAttribute attr[2] = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The plan grid: CTA 0 plans, CTAs 1..p.write_ctas write the new tokens' K/V rows.
// With `dependent` it may become resident while the previous grid in the stream
// runs (it waits for that grid on the device before reading anything).
cudaError_t launch_plan(const PlanParams& p, cudaStream_t s, bool dependent);
// One warp waits on an mbarrier that nothing completes until the bounded wait
// gives up and sets the timeout bit in *err (failure-detection self-test).
cudaError_t launch_wait_selftest(int* err, cudaStream_t s);
// Key sums and V maxima, then the K, V and Q codes that QuantParams asks for.
cudaError_t launch_quant(const QuantParams& p, int sms, cudaStream_t s);
// head_dim 128: `to` is the output map (bf16 [total_q][n_heads_q][128] as
// [128, G, n_heads_kv, total_q], box [32, G, 1, T], 64-byte swizzle), through
// which the kernel stores full q tiles; unused at head_dim 256.
cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tkv,
                             const CUtensorMap& to, int head_dim, int grid, cudaStream_t s, bool dependent);
// Quantised-QK prefill (head_dim 128): tq8 over the e4m3 Q codes, tk8 over the
// e4m3 K blocks, tkv over the bf16 cache (V).
cudaError_t launch_attention_fp8(const AttnParams& p, const CUtensorMap& tq8, const CUtensorMap& tk8,
                                 const CUtensorMap& tkv, const CUtensorMap& to, int grid, cudaStream_t s,
                                 bool dependent);
// fp8 P.V prefill (head_dim 128): as above, with tv8 over the transposed e4m3
// V tiles [tiles][n_heads_kv][128 channels][128 keys] in place of the bf16 V.
cudaError_t launch_attention_fp8pv(const AttnParams& p, const CUtensorMap& tq8, const CUtensorMap& tk8,
                                   const CUtensorMap& tv8, const CUtensorMap& to, int grid, cudaStream_t s,
                                   bool dependent);
// head_dim 128 with two q tiles per CTA (bf16): items of two q tiles from a plan
// made with PlanParams::pair; `to` as for launch_attention.
cudaError_t launch_attention_2q(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tkv,
                                const CUtensorMap& to, int grid, cudaStream_t s, bool dependent);
cudaError_t attention2q_set_attributes();
// head_dim 256 with CTA pairs (cta_group::2 MMAs, 128-key tiles): items of two
// q tiles from a plan made with PlanParams::pair; grid even.
cudaError_t launch_attention_pair(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tkv,
                                  int grid, cudaStream_t s, bool dependent);
cudaError_t launch_decode(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tkv,
                          int head_dim, int grid, cudaStream_t s, bool dependent);
size_t decode_smem_bytes(int head_dim);
cudaError_t decode_set_attributes();
// Keys per KV tile of the prefill kernel (head_dim 256: 128 with CTA pairs, else 64).
int attention_block_n(int head_dim, bool pair = false);
size_t attention_smem_bytes(int head_dim);
cudaError_t attention_set_attributes();

}  // namespace pattn
