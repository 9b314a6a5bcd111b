/*
 * pattn.h -- C ABI of libpattn: paged-KV varlen attention on GB300 (sm_103a).
 *
 * The operation (one call computes it for a whole batch):
 *
 *   for every sequence b, query token i < ql_b = cu_q[b+1] - cu_q[b], query head h:
 *     hk  = h / (n_heads_q / n_heads_kv)             contiguous GQA groups
 *     pos = L_b - ql_b + i                           queries are the last ql_b keys
 *     J   = { j < L_b : !causal or j <= pos }
 *     out[cu_q[b]+i][h] = sum_{j in J} softmax_j(scale * q . k_j) v_j   (0 if J is empty)
 *
 * with k_j, v_j row j % page_size of page block_table[b][j / page_size] of the
 * pool. Sources: the trtllm-gen paged decode manifest (examples/decode.json:
 * op "decode" parameters out, q, k, v, table, seq, cuq, seqs, tokens; the
 * scratch buffers "partial" and "stats" of its split-KV launch; its Q and
 * K/V tensor maps, which fix the GQA packing and the page geometry) and the
 * FlashAttention-4 SM100MHA2Q kernel doc (paged KV lookup, causal or unmasked
 * mask, ragged valid lengths, KV partitions). Q/K/V/out are bf16; scores,
 * softmax and accumulation are fp32.
 *
 * Conventions for every call:
 *   - Device pointers are owned by the caller; the library keeps none of them
 *     past the call. Calls are asynchronous and ordered on `stream`; nothing
 *     here synchronises the host except pattn_get_device_status,
 *     pattn_profile_read, pattn_profile_read_kernels and pattn_forward_host.
 *   - Errors the host can see (null or misaligned pointers, sizes, unsupported
 *     shapes) are returned before anything is launched.
 *   - Errors only the data shows (a block-table entry outside the pool inside
 *     a live range, lengths beyond the host bounds, cu_q out of order) set a
 *     device error word and zero the affected sequence's output rows; no call
 *     traps or reads outside the pool. pattn_get_device_status reports them.
 *   - Every wait inside a kernel is bounded (about 2 s); a wait that runs out
 *     sets the error word (PATTN_ERR_DEVICE_TIMEOUT) and the kernel returns.
 *   - The library is not re-entrant across host threads for one device (one
 *     workspace per device).
 */
#ifndef PATTN_H_
#define PATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the two types are the same pointer); NULL = legacy default stream. */
typedef struct CUstream_st *pattn_stream_t;

typedef enum pattn_status {
  PATTN_OK = 0,
  PATTN_ERR_INVALID_ARG = 1,      /* null/misaligned pointer, bad size or bound */
  PATTN_ERR_UNSUPPORTED = 2,      /* head_dim not 128/256, page_size not 64, group > 128, ... */
  PATTN_ERR_CUDA = 3,             /* a CUDA runtime/driver call failed */
  PATTN_ERR_NO_MEMORY = 4,        /* workspace allocation failed or caller workspace too small */
  PATTN_ERR_DEVICE_BAD_INPUT = 5, /* device data rejected (page index, lengths, cu_q) */
  PATTN_ERR_DEVICE_TIMEOUT = 6    /* a bounded wait inside a kernel ran out */
} pattn_status;

/*
 * pattn_forward -- causal or full attention over a paged (or contiguous) KV cache.
 *
 *   out         bf16 [total_q][n_heads_q][head_dim], written in full.
 *   q           bf16 [total_q][n_heads_q][head_dim].
 *   kv_pool     paged:      bf16 [num_pages][2 (K, V)][page_size][n_heads_kv][head_dim];
 *               contiguous: bf16 [2 (K, V)][num_pages][n_heads_kv][head_dim] when
 *               block_table is NULL (num_pages then counts rows of each plane, and
 *               sequence b's keys are rows sum(seq_lens[0..b)) onwards).
 *   block_table int32 [num_seqs][ceil(max_kv / page_size)]: the page of each
 *               logical slot; slots at or past ceil(L_b / page_size) are never
 *               read (-1 by convention). NULL selects the contiguous cache.
 *   seq_lens    int32 [num_seqs]: KV length L_b, the current queries included.
 *   cu_q        int32 [num_seqs + 1]: query offsets, cu_q[0] = 0, non-decreasing,
 *               cu_q[num_seqs] = total_q.
 *   num_seqs, total_q   batch size and number of query tokens (the manifest's
 *               "seqs" and "tokens" op parameters).
 *   max_q, max_kv       host upper bounds of ql_b and L_b (size the plan and the
 *               block-table row stride).
 *   n_heads_q, n_heads_kv, head_dim, page_size   head_dim in {128, 256},
 *               page_size 64, n_heads_q a multiple of n_heads_kv, group <= 128.
 *   num_pages   pages in the pool (bounds every block-table entry).
 *   scale       softmax scale, finite and >= 0.
 *   causal      0: every key of the sequence; 1: keys up to the query position.
 *   stream      stream the launches go on: the plan, then the decode kernel (units
 *               of at most 16 packed query rows; not launched when the bounds rule
 *               such units out, i.e. every sequence holds at least
 *               total_q - (num_seqs - 1) * max_q > 16 / group queries) and/or the
 *               prefill kernel (every other unit).
 *
 * All pointers 16-byte aligned. The first call on a device allocates the
 * library workspace (grow-only) unless pattn_set_workspace gave one.
 *
 * CUDA graphs: once the workspace is large enough for the bounds (a first
 * call outside the capture, or pattn_set_workspace), a call only launches
 * kernels on `stream` and can be captured. The plan is made on the device at
 * every replay, from whatever the length, offset and table buffers hold then,
 * within the bounds given at capture.
 */
pattn_status pattn_forward(void *out, const void *q, const void *kv_pool,
                           const int32_t *block_table, const int32_t *seq_lens,
                           const int32_t *cu_q, int num_seqs, int total_q, int max_q,
                           int max_kv, int n_heads_q, int n_heads_kv, int head_dim,
                           int page_size, int num_pages, float scale, int causal,
                           pattn_stream_t stream);

/*
 * pattn_forward_append -- the cache write in front of attention, then
 * pattn_forward: the `reshape_and_cache_flash` (kv_write) node that comes right
 * before `attend` in the GB10 model graph, in the same stream-ordered call.
 *
 *   k_new, v_new  bf16 [total_q][n_heads_kv][head_dim]: the K and V rows of the
 *                 query tokens, in the token order of q.
 *   kv_pool       as for pattn_forward, written: token i of sequence b
 *                 (i < ql_b) goes to cache position L_b - ql_b + i, i.e. row
 *                 (pos mod page_size) of page block_table[b][pos / page_size]
 *                 (contiguous cache: row sum(seq_lens[0..b)) + pos of the K and
 *                 V planes). Nothing else in the pool is written.
 *   other arguments as for pattn_forward; seq_lens count the new tokens.
 *
 * The write runs in the plan kernel's grid (CTAs beyond the planning one, a
 * warp per new token) while the plan is made, so it costs no launch of its
 * own; the attention kernels then read the updated cache. Tokens at positions
 * < 0 (more queries than keys) are not written. Sequences rejected on the device
 * (PATTN_ERR_DEVICE_BAD_INPUT) are neither written nor attended (rows zero).
 * k_new and v_new are caller-owned device buffers, 16-byte aligned; they must
 * not overlap kv_pool.
 */
pattn_status pattn_forward_append(void *out, const void *q, const void *k_new, const void *v_new,
                                  void *kv_pool, const int32_t *block_table,
                                  const int32_t *seq_lens, const int32_t *cu_q, int num_seqs,
                                  int total_q, int max_q, int max_kv, int n_heads_q,
                                  int n_heads_kv, int head_dim, int page_size, int num_pages,
                                  float scale, int causal, pattn_stream_t stream);

/*
 * pattn_forward_fp8qk -- the quantised-QK variant: SageAttention2's preparation
 * phases as on the GB10 "sage2" benchmark page (K-mean smoothing, Q and K
 * quantisation; phases k_mean_and_smoothing_preparation, q_int8_quantization,
 * k_int8_subtract_mean_quantization), with e4m3 codes instead of int8 (on this
 * part the e4m3 tensor rate is twice the bf16 one and the int8 rate is far
 * below it), then attention with S = Q K^T from e4m3 codes and O = P V in bf16.
 * Same arguments and output as pattn_forward; head_dim 128 only.
 *
 *   K is smoothed per (sequence, KV head, channel) by its mean over the
 *   sequence's keys (the softmax cancels the shift), summed exactly in fixed
 *   point: each key clamped to +-1024 and rounded to a multiple of 2^-32, then
 *   sum * 2^-32 / L in float64, rounded to fp32; each 64-key block of a
 *   sequence and KV head gets one scale, each query row (token, head) one:
 *   scale = amax / 448, code = e4m3 round-to-nearest-even of x / scale,
 *   saturated. The result is attention over the dequantised Q and K.
 *   Units of at most 16 packed query rows (decode) take the bf16 decode kernel.
 *   Needs pattn_workspace_size_fp8qk bytes of workspace. PATTN_ERR_UNSUPPORTED
 *   for head_dim != 128 or max_kv > 2^20.
 */
pattn_status pattn_forward_fp8qk(void *out, const void *q, const void *kv_pool,
                                 const int32_t *block_table, const int32_t *seq_lens,
                                 const int32_t *cu_q, int num_seqs, int total_q, int max_q,
                                 int max_kv, int n_heads_q, int n_heads_kv, int head_dim,
                                 int page_size, int num_pages, float scale, int causal,
                                 pattn_stream_t stream);

/*
 * pattn_quantize_qk -- only the codes and scales of pattn_forward_fp8qk, into
 * caller-owned device buffers (nb = 2 * ceil(max_kv / 128)):
 *
 *   q8       e4m3 bytes [total_q][n_heads_q][128], 16-byte aligned
 *   q_scale  fp32 [total_q][n_heads_q]
 *   k8       e4m3 bytes [num_seqs * nb][64][n_heads_kv][128], 16-byte aligned:
 *            64-key block j of sequence b is block b * nb + j; key rows past
 *            L_b in its last block are zero; later blocks are not written
 *   k_scale  fp32 [num_seqs * nb][n_heads_kv] (written for the same blocks)
 *
 * Other arguments as for pattn_forward. Rejected sequences (device error word)
 * are not written.
 */
pattn_status pattn_quantize_qk(void *q8, float *q_scale, void *k8, float *k_scale, const void *q,
                               const void *kv_pool, const int32_t *block_table,
                               const int32_t *seq_lens, const int32_t *cu_q, int num_seqs,
                               int total_q, int max_q, int max_kv, int n_heads_q, int n_heads_kv,
                               int head_dim, int page_size, int num_pages, pattn_stream_t stream);

/* Workspace bytes pattn_forward_fp8qk needs for these bounds (0 if unsupported). */
size_t pattn_workspace_size_fp8qk(int num_seqs, int total_q, int max_q, int max_kv, int n_heads_q,
                                  int n_heads_kv, int head_dim, int page_size);

/*
 * pattn_forward_fp8 -- pattn_forward_fp8qk with P and V in e4m3 as well: the V
 * phases of the same GB10 "sage2" page (v_fp8_transpose_scale_quantization:
 * transpose/pad/permute and scale/fp8; v_scale_fp8_quantization), then
 * O = P V as e4m3 MMAs with fp32 accumulation. Same arguments and output as
 * pattn_forward; head_dim 128 and max_kv <= 2^20 only (else
 * PATTN_ERR_UNSUPPORTED). Needs pattn_workspace_size_fp8 bytes of workspace.
 *
 *   V: one scale per (sequence, KV head, channel), scale = amax / 448 over the
 *   sequence's keys, code = e4m3 of v * (448 / amax) as for Q and K, stored
 *   transposed (keys innermost) in zero-padded 128-key tiles. P: e4m3 of
 *   p * 2^2 with p taken against a running row max that the tile's codes never
 *   exceed 2^8 under, so no code saturates; the row sum is the fp32 sum of the
 *   unrounded p. The output is the attention over the dequantised Q, K and V
 *   up to the rounding of P: per element at most
 *   (2^-4 sum_j p_j |v_j| + 2^-12 sum_j |v_j|) / sum_j p_j
 *   (p relative to the row max, v the dequantised V) plus the bf16 rounding of
 *   the output. Units of at most 16 packed query rows take the bf16 decode kernel.
 */
pattn_status pattn_forward_fp8(void *out, const void *q, const void *kv_pool,
                               const int32_t *block_table, const int32_t *seq_lens,
                               const int32_t *cu_q, int num_seqs, int total_q, int max_q,
                               int max_kv, int n_heads_q, int n_heads_kv, int head_dim,
                               int page_size, int num_pages, float scale, int causal,
                               pattn_stream_t stream);

/*
 * pattn_quantize_v -- only the V codes and scales of pattn_forward_fp8, into
 * caller-owned device buffers (nb = 2 * ceil(max_kv / 128)):
 *
 *   v8       e4m3 bytes [num_seqs * nb / 2][n_heads_kv][128 channels][128 keys],
 *            16-byte aligned: 128-key tile t of sequence b is tile b * nb / 2 + t;
 *            keys past L_b in its last tile are zero codes; later tiles are
 *            not written
 *   v_scale  fp32 [num_seqs][n_heads_kv][128], 16-byte aligned
 *
 * Other arguments as for pattn_forward (no queries are read). Rejected
 * sequences (device error word) are not written.
 */
pattn_status pattn_quantize_v(void *v8, float *v_scale, const void *kv_pool,
                              const int32_t *block_table, const int32_t *seq_lens,
                              const int32_t *cu_q, int num_seqs, int total_q, int max_q, int max_kv,
                              int n_heads_q, int n_heads_kv, int head_dim, int page_size,
                              int num_pages, pattn_stream_t stream);

/* Workspace bytes pattn_forward_fp8 needs for these bounds (0 if unsupported). */
size_t pattn_workspace_size_fp8(int num_seqs, int total_q, int max_q, int max_kv, int n_heads_q,
                                int n_heads_kv, int head_dim, int page_size);

/*
 * pattn_selftest_wait_timeout -- failure-detection self-test: launches one warp
 * that waits, with the attention kernels' bounded-wait code, on an mbarrier
 * phase that nothing completes. After the wait limit (2 s) it sets the timeout
 * bit of the device error word and returns; nothing faults or hangs, and the
 * context stays usable. The next pattn_get_device_status on the stream returns
 * PATTN_ERR_DEVICE_TIMEOUT. Returns the launch status.
 */
pattn_status pattn_selftest_wait_timeout(pattn_stream_t stream);

/*
 * pattn_selftest_attention_timeout -- failure-detection self-test of the
 * attention kernels' own abort path. Runs pattn_forward on the given batch
 * (same arguments and rules) with one change: in each attention kernel the
 * batch launches that has work (the swap-AB decode kernel, the one-q-tile and
 * two-q-tile prefill kernels), the first CTA's MMA-issuing thread first waits for a
 * barrier phase that nothing completes before that thread's own drain. After
 * the wait limit (about 2 s) the wait gives up: it sets the timeout bit of the
 * device error word and the CTA's abort flag; every role of the CTA then
 * leaves its loop, waits (bounded) for the copies and MMAs it has in flight,
 * frees its tensor memory and exits. Nothing faults or hangs, and the context
 * stays usable: the next pattn_get_device_status returns
 * PATTN_ERR_DEVICE_TIMEOUT and later calls run normally. The output rows of
 * the first CTA's items are unspecified. Batches that take the CTA-pair
 * prefill kernel (head_dim 256 with two q tiles per sequence) return
 * PATTN_ERR_UNSUPPORTED. Returns the launch status.
 */
pattn_status pattn_selftest_attention_timeout(void *out, const void *q, const void *kv_pool,
                                              const int32_t *block_table, const int32_t *seq_lens,
                                              const int32_t *cu_q, int num_seqs, int total_q, int max_q,
                                              int max_kv, int n_heads_q, int n_heads_kv, int head_dim,
                                              int page_size, int num_pages, float scale, int causal,
                                              pattn_stream_t stream);

/*
 * The tile plan of a batch, for inspection (tests): runs only the device-side
 * planner that pattn_forward launches first (step "plan / tile scheduler" of
 * the method: varlen q tiles of T = 128 / G tokens with GQA packing, causal
 * tile skipping as the FlashAttention-4 kernel doc's mask_status describes,
 * KV splits of single-q-tile units as the decode manifest's MultiCtasKv),
 * then copies its two work lists to host memory and synchronises `stream`.
 *
 * Arguments as pattn_forward (no Q, cache or output pointers; scale is not
 * needed). prefill_items / decode_items: host int32 [capacity][4] each,
 * written with the first min(count, capacity) items of the head_dim-specific
 * prefill kernel's list and of the swap-AB decode kernel's list, in list
 * order (longest first). counts: host int32[4] = {prefill items, decode items,
 * split units, partial rows}.
 *
 * Item record {x, y, z, w}: x = sequence | split << 24; y = kv_head << 16 |
 * q tile (the first of an item's two q tiles: CTA pairs at head_dim 256, the
 * two-q-tile kernel for non-causal head_dim 128); z = first KV
 * tile << 16 | end KV tile (tiles of 128 keys, or 64 for the one-CTA
 * head_dim-256 prefill kernel); w = first partial row of a split item, -1
 * otherwise. Returns PATTN_ERR_NO_MEMORY if the plan did not fit the
 * workspace; errors as pattn_forward otherwise.
 */
pattn_status pattn_plan_items(const int32_t *block_table, const int32_t *seq_lens, const int32_t *cu_q,
                              int num_seqs, int total_q, int max_q, int max_kv, int n_heads_q,
                              int n_heads_kv, int head_dim, int page_size, int num_pages, int causal,
                              int32_t *prefill_items, int32_t *decode_items, int capacity,
                              int32_t *counts, pattn_stream_t stream);

/* Bytes of the fixed device scratch behind pattn_forward_noalloc. */
#define PATTN_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * pattn_forward_noalloc -- pattn_forward without any allocation. The pages
 * have no counterpart of this entry point; it exists for callers that must
 * not allocate device memory: a serving process whose caching allocator has
 * already reserved nearly all of the GPU (a fresh cudaMalloc would fail or
 * force the cache to be emptied), a decode loop that cannot afford the device
 * synchronisation cudaMalloc/cudaFree imply, or a host application that owns
 * every device buffer itself.
 *
 * Same arguments, layouts and results as pattn_forward. Instead of the
 * library workspace it uses one fixed device array of
 * PATTN_NOALLOC_SCRATCH_BYTES, compiled into the library: every GPU that
 * loads the library holds it until the process exits. Nothing here calls
 * cudaMalloc, cudaFree or any allocating routine.
 *
 * Acceptance: the work list and split-KV scratch a batch can need are bounded
 * from num_seqs, total_q, max_q, max_kv, the heads and the device's SM count
 * (at most 64 splits per (sequence, KV head) unit, and at most ceil(max_kv /
 * 64); per kernel list at most the planner's item target plus its units).
 * A batch whose bound exceeds the array is rejected with PATTN_ERR_NO_MEMORY
 * before anything is launched. The bound never exceeds pattn_workspace_size
 * for the same arguments, so every batch whose pattn_workspace_size fits is
 * accepted; some larger ones (short max_kv) are accepted too. For example,
 * 64 sequences x 32/8 heads, head_dim 128, one query each and up to 8k keys
 * fit.
 *
 * The first call on a device sets the scratch up (looks up its device
 * address and clears its header, a synchronous step), so make that first call
 * before any stream capture. All calls share the one array and it keeps the
 * previous call's contents: calls that overlap on the GPU (other streams,
 * other host threads) race on it and must be serialised by the caller.
 * Device-side data errors (a rejected page or length, a wait that ran out)
 * set the scratch's own error word; pattn_get_device_status reads and clears
 * it together with the workspace's. Rejected rows are zero-filled.
 */
pattn_status pattn_forward_noalloc(void *out, const void *q, const void *kv_pool,
                                   const int32_t *block_table, const int32_t *seq_lens,
                                   const int32_t *cu_q, int num_seqs, int total_q, int max_q,
                                   int max_kv, int n_heads_q, int n_heads_kv, int head_dim,
                                   int page_size, int num_pages, float scale, int causal,
                                   pattn_stream_t stream);

/*
 * pattn_forward_host -- the same operation on HOST buffers, end to end: copies
 * the inputs to device buffers the library keeps (grow-only, per device),
 * runs pattn_forward on `stream`, copies `out` back and synchronises the
 * stream. Layouts and arguments as for pattn_forward. Host buffers should be
 * pinned for full copy bandwidth. kv_pool_bytes is the size of the pool buffer.
 */
pattn_status pattn_forward_host(void *out, const void *q, const void *kv_pool,
                                size_t kv_pool_bytes, const int32_t *block_table,
                                const int32_t *seq_lens, const int32_t *cu_q, int num_seqs,
                                int total_q, int max_q, int max_kv, int n_heads_q,
                                int n_heads_kv, int head_dim, int page_size, int num_pages,
                                float scale, int causal, pattn_stream_t stream);

/*
 * Workspace bytes pattn_forward needs for these bounds: a header with the
 * device error word, the planned work list, the split-KV partial O and
 * (max, sum) scratch and the per-unit finished-split counters (the manifest's
 * "partial", "stats" and "counter" buffers).
 */
size_t pattn_workspace_size(int num_seqs, int total_q, int max_q, int max_kv, int n_heads_q,
                            int n_heads_kv, int head_dim, int page_size);

/*
 * Use caller-owned device memory as the workspace of the current device
 * (ptr 256-byte aligned; NULL returns to the library-owned one). The library
 * clears its header once here; later calls need at least pattn_workspace_size
 * bytes or return PATTN_ERR_NO_MEMORY.
 */
pattn_status pattn_set_workspace(void *ptr, size_t bytes);

/*
 * Synchronises `stream`, reads and clears the device error words of the
 * current device (the workspace's, and that of the fixed scratch behind
 * pattn_forward_noalloc once it is set up). Allocates nothing. Returns
 * PATTN_OK, PATTN_ERR_DEVICE_BAD_INPUT or PATTN_ERR_DEVICE_TIMEOUT (timeout
 * wins if both are set).
 */
pattn_status pattn_get_device_status(pattn_stream_t stream);

/* Static description of a status code. */
const char *pattn_status_string(pattn_status status);

/*
 * Kernel timing: while enabled, pattn_forward records CUDA events around each
 * of its launches on its stream (at most 4096 calls are kept).
 * pattn_profile_read synchronises those events and returns the summed device
 * time in milliseconds of the plan kernel and of the attention kernels
 * (decode and prefill) and the number of calls recorded, then clears the
 * record. ms_combine is the time after the attention kernels; split-KV
 * partials are merged inside them, so it is close to zero.
 */
pattn_status pattn_profile_enable(int on);
pattn_status pattn_profile_read(double *ms_plan, double *ms_attention, double *ms_combine,
                                int *calls);

/*
 * The same record split by kernel: ms[0] plan (with the cache write of
 * pattn_forward_append, which runs in the plan's grid), ms[1] quantisation
 * passes (pattn_forward_fp8qk, pattn_forward_fp8), ms[2] decode kernel, ms[3]
 * prefill kernel, ms[4] time after the attention kernels (nothing runs there:
 * both merge their own splits). ms holds 5 doubles. Clears the record like
 * pattn_profile_read.
 */
pattn_status pattn_profile_read_kernels(double *ms, int *calls);

#ifdef __cplusplus
}
#endif

#endif /* PATTN_H_ */
