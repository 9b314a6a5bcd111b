// api.cu -- host side of libpattn: argument validation, per-device workspace,
// TMA tensor-map encoding and the launch sequence plan (whose grid also writes
// the new tokens' K/V rows for pattn_forward_append) -> (quantisation) ->
// decode -> prefill (both attention kernels merge their own split-KV partials).
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/pattn.h"
#include "kernels.cuh"

namespace pattn {
namespace {

constexpr int kMaxDevices = 64;
// Split target: about 2 items per SM in each kernel's list (in halves). Fewer,
// longer items cost less pipeline start-up; a unit is split only when it holds
// more than about half an SM's share of its kernel's work (measured: decode
// batch 0.200 -> 0.1855 ms against 4 items per SM of the whole job's work; its
// units longer than ~7.7k keys still take the split-KV path).
constexpr int kTargetHalfItemsPerSm = 4;
// Most items per kernel list the split heuristic may aim at (the workspace
// bound below assumes it when the device is not known).
constexpr int kTargetItemsCap = 512;
constexpr int kMinChunk = 16;          // 64-key blocks per split, at least (split and merge cost more than short items save below this)
constexpr int kProfileCap = 4096;
constexpr int kPlanWarps = 32;         // warps of a plan-grid CTA (one new token each when writing)

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Events around plan | cache write / quantisation | decode kernel | prefill
// kernel | (the former merge slot, now empty).
struct ProfileRec {
  cudaEvent_t ev[6];
};

struct DeviceState {
  bool ready = false;
  int sms = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  bool ws_caller = false;
  void* stage[6] = {};
  size_t stage_bytes[6] = {};
  std::vector<ProfileRec> prof;
  std::vector<ProfileRec> prof_pool;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
bool g_profile = false;

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }

struct Shape {
  int group, tokens_per_tile, block_n;
  bool pair;   // head_dim 256 prefill on CTA pairs (some sequence may have two q tiles)
  bool two_q;  // head_dim 128 bf16 non-causal prefill with two q tiles per CTA (same condition)
};

// The batch description and head configuration (everything but the Q, K/V and
// output pointers); fills the tiling of the batch.
pattn_status check_shape(const int32_t* bt, const int32_t* seq_lens, const int32_t* cu_q, int num_seqs,
                         int total_q, int max_q, int max_kv, int hq, int hkv, int d, int page,
                         int num_pages, float scale, int causal, Shape* sh) {
  if (!seq_lens || !cu_q) return PATTN_ERR_INVALID_ARG;
  if (!aligned(seq_lens, 4) || !aligned(cu_q, 4) || (bt && !aligned(bt, 4)))
    return PATTN_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_q < 0 || max_q < 0 || max_kv < 0) return PATTN_ERR_INVALID_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return PATTN_ERR_INVALID_ARG;
  if (num_pages <= 0) return PATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return PATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PATTN_ERR_INVALID_ARG;
  if (scale < 0.f) return PATTN_ERR_UNSUPPORTED;
  if (d != 128 && d != 256) return PATTN_ERR_UNSUPPORTED;
  if (page != kPage) return PATTN_ERR_UNSUPPORTED;
  const int g = hq / hkv;
  if (g > kBM) return PATTN_ERR_UNSUPPORTED;
  sh->group = g;
  sh->tokens_per_tile = kBM / g;
  sh->pair = d == 256 && max_q > sh->tokens_per_tile;
  // Two q tiles per CTA at head_dim 128 for non-causal batches only: measured
  // on the 37,810-token batch it runs 8-11 % faster at the power limit (each K/V
  // tile is loaded once per q tile pair, so the part holds a higher clock); on
  // causal batches (short items along the triangle) the one-q-tile kernel is
  // as fast at the power limit and about 18 % faster per clock cycle.
  sh->two_q = d == 128 && causal == 0 && max_q > sh->tokens_per_tile;
  sh->block_n = attention_block_n(d, sh->pair);
  // item encoding keeps q tiles and KV tiles in 16 bits
  if (cdiv(max_q, sh->tokens_per_tile) > 65535) return PATTN_ERR_UNSUPPORTED;
  if (cdiv(max_kv, sh->block_n) > 65535) return PATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_pages) * 2 > 0x7fffffffLL) return PATTN_ERR_UNSUPPORTED;
  if (num_seqs > kSeqMask) return PATTN_ERR_UNSUPPORTED;  // item encoding: 24-bit sequence index
  if (static_cast<long long>(total_q) * hq * d > (1LL << 40)) return PATTN_ERR_UNSUPPORTED;
  return PATTN_OK;
}

pattn_status check_args(const void* out, const void* q, const void* kv, const int32_t* bt,
                        const int32_t* seq_lens, const int32_t* cu_q, int num_seqs, int total_q,
                        int max_q, int max_kv, int hq, int hkv, int d, int page, int num_pages,
                        float scale, int causal, Shape* sh) {
  if (!out || !q || !kv) return PATTN_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(kv, 16)) return PATTN_ERR_INVALID_ARG;
  return check_shape(bt, seq_lens, cu_q, num_seqs, total_q, max_q, max_kv, hq, hkv, d, page, num_pages,
                     scale, causal, sh);
}

struct WsLayout {
  size_t hdr, seq_info, seq_plan, seq_part, items, dec_items, unit_cnt, part_ml, part_o, total;
  int max_items, max_units, max_part_rows;
};

// Items per list the planner aims at on a device with `sms` SMs; the decode
// list may take up to a quarter more (the planner chooses per call).
inline int plan_target(int sms) { return std::min(kTargetHalfItemsPerSm * sms / 2, kTargetItemsCap * 4 / 5); }
inline int plan_target_max(int sms) { return plan_target(sms) + plan_target(sms) / 4; }

// Workspace layout for these bounds. `target` is the planner's item target per
// list (kTargetItemsCap when the device is not known). The planner sizes the
// splits of each of its two lists (decode kernel, prefill kernel) from that
// list's own work, so each list holds at most target + its units splits:
// 2 * target + units in all. With max_kv >= 0 the split bound also uses the
// planner's per-unit limit (at most min(kMaxSplits, ceil(max_kv/64)) splits
// per unit).
WsLayout ws_layout(int num_seqs, int total_q, int max_q, int hq, int hkv, int d, int max_kv = -1,
                   int target = kTargetItemsCap) {
  WsLayout w{};
  const int g = hq / hkv;
  const int T = kBM / g;
  const long long units = static_cast<long long>(num_seqs) * hkv;
  const long long qtiles = cdiv(total_q, T) + static_cast<long long>(num_seqs);
  // per list: one item per (q tile, KV head), a split unit's S splits in place of its one
  const long long items = static_cast<long long>(hkv) * qtiles + target + units + 64;
  const long long rows_cap = std::min<long long>(kBM, static_cast<long long>(max_q) * g);
  long long splits = 2LL * target + units;
  if (max_kv >= 0) {
    const long long per_unit = std::min<long long>(kMaxSplits, std::max(1, cdiv(max_kv, kPage)));
    splits = std::min(splits, units * per_unit);
  }
  const long long part_rows = splits * std::max<long long>(rows_cap, 1);
  w.max_items = static_cast<int>(std::min<long long>(items, 0x7fffffffLL));
  w.max_units = static_cast<int>(std::min<long long>(units, 0x7fffffffLL));
  w.max_part_rows = static_cast<int>(std::min<long long>(part_rows, 0x7fffffffLL));
  size_t off = 0;
  w.hdr = off;
  off += kHdrWords * sizeof(int);
  w.seq_info = off = align_up(off, 256);
  off += sizeof(int4) * static_cast<size_t>(num_seqs);
  w.seq_plan = off = align_up(off, 256);
  off += sizeof(int4) * static_cast<size_t>(num_seqs);
  w.seq_part = off = align_up(off, 256);
  off += sizeof(int) * static_cast<size_t>(num_seqs);
  w.items = off = align_up(off, 256);
  off += sizeof(int4) * static_cast<size_t>(w.max_items);
  w.dec_items = off = align_up(off, 256);
  off += sizeof(int4) * static_cast<size_t>(w.max_items);
  w.unit_cnt = off = align_up(off, 256);
  off += sizeof(int) * static_cast<size_t>(w.max_units);
  w.part_ml = off = align_up(off, 256);
  off += sizeof(float2) * static_cast<size_t>(w.max_part_rows);
  w.part_o = off = align_up(off, 256);
  off += sizeof(float) * static_cast<size_t>(d) * static_cast<size_t>(w.max_part_rows);
  w.total = align_up(off, 256);
  return w;
}

pattn_status cuda_fail(cudaError_t e) {
  if (e == cudaSuccess) return PATTN_OK;
  if (e == cudaErrorMemoryAllocation) return PATTN_ERR_NO_MEMORY;
  return PATTN_ERR_CUDA;
}

// Per-device one-time set-up; caller holds g_mu.
pattn_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return PATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PATTN_ERR_UNSUPPORTED;
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PATTN_ERR_CUDA;
    if (major != 10 || minor != 3) return PATTN_ERR_UNSUPPORTED;  // built for sm_103a only
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return PATTN_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (attention_set_attributes() != cudaSuccess) return PATTN_ERR_CUDA;
    if (attention2q_set_attributes() != cudaSuccess) return PATTN_ERR_CUDA;
    if (decode_set_attributes() != cudaSuccess) return PATTN_ERR_CUDA;
    st.ready = true;
  }
  *out = &st;
  return PATTN_OK;
}

pattn_status ensure_workspace(DeviceState& st, size_t need) {
  if (st.ws_caller) return st.ws_bytes >= need ? PATTN_OK : PATTN_ERR_NO_MEMORY;
  if (st.ws && st.ws_bytes >= need) return PATTN_OK;
  if (st.ws) {
    // grow: the old buffer may still be in use by queued work
    cudaDeviceSynchronize();
    cudaFree(st.ws);
    st.ws = nullptr;
    st.ws_bytes = 0;
  }
  size_t bytes = align_up(need + need / 4, 1 << 20);
  cudaError_t e = cudaMalloc(&st.ws, bytes);
  if (e != cudaSuccess) {
    st.ws = nullptr;
    return cuda_fail(e);
  }
  e = cudaMemset(st.ws, 0, kHdrWords * sizeof(int));
  if (e != cudaSuccess) return PATTN_ERR_CUDA;
  st.ws_bytes = bytes;
  return PATTN_OK;
}

pattn_status encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                    const cuuint64_t* strides, const cuuint32_t* box,
                    CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, dtype, static_cast<cuuint32_t>(rank),
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PATTN_OK : PATTN_ERR_CUDA;
}

// Longest sequence of the quantised-QK path: the fixed-point key sums (units of
// 2^-32, values clamped to +-1024) stay below 2^62 in magnitude.
constexpr int kFp8MaxKv = 1 << 20;

// Workspace regions of the quantised variants, after the regular ones (see
// QuantParams for the layouts; the V regions only with_v). nb_max is even, so
// that both key halves of a 128-key tile have a block.
struct Fp8Layout {
  size_t k_sum, q8, q_scale, k8, k_scale, v8, v_scale, total;  // k_sum: the quant_scratch_bytes region
  int nb_max;
};
Fp8Layout fp8_layout(size_t base, int num_seqs, int total_q, int max_kv, int hq, int hkv, int d,
                     bool with_v = false) {
  Fp8Layout f{};
  f.nb_max = 2 * std::max(1, cdiv(max_kv, 2 * kPage));
  const size_t B = static_cast<size_t>(num_seqs), nb = static_cast<size_t>(f.nb_max);
  size_t off = align_up(base, 256);
  f.k_sum = off;
  off += quant_scratch_bytes(num_seqs, hkv, d);
  f.q8 = off = align_up(off, 256);
  off += static_cast<size_t>(total_q) * hq * d;
  f.q_scale = off = align_up(off, 256);
  off += static_cast<size_t>(total_q) * hq * sizeof(float);
  f.k8 = off = align_up(off, 256);
  off += B * nb * kPage * hkv * d;
  f.k_scale = off = align_up(off, 256);
  off += B * nb * hkv * sizeof(float);
  if (with_v) {
    f.v8 = off = align_up(off, 256);
    off += B * (nb / 2) * hkv * d * 128;
    f.v_scale = off = align_up(off, 256);
    off += B * hkv * d * sizeof(float);
  }
  f.total = align_up(off, 256);
  return f;
}

// What one call computes: attention (bf16), attention with e4m3 Q/K codes,
// attention with e4m3 Q/K/P/V codes, or only codes (those QuantBufs names).
enum class Mode { kBf16, kFp8, kFp8Pv, kQuantOnly, kPlanOnly };

// Device buffers of the e4m3 codes (workspace regions or caller buffers).
struct QuantBufs {
  uint8_t* q8 = nullptr;
  float* q_scale = nullptr;
  uint8_t* k8 = nullptr;
  float* k_scale = nullptr;
  uint8_t* v8 = nullptr;
  float* v_scale = nullptr;
  void* scratch = nullptr;  // quant_scratch_bytes
  int nb_max = 0;
};

ProfileRec take_events(DeviceState& st) {
  ProfileRec r{};
  if (!st.prof_pool.empty()) {
    r = st.prof_pool.back();
    st.prof_pool.pop_back();
    return r;
  }
  for (auto& e : r.ev) cudaEventCreate(&e);
  return r;
}

// Encodes the tensor maps and launches plan (+ cache write in the same grid) ->
// [quantisation] -> decode -> prefill with the workspace at `wsb` (laid out as
// L); the attention kernels merge their own KV splits. Caller holds g_mu.
pattn_status launch_all(DeviceState& st, uint8_t* wsb, const WsLayout& L, void* out, const void* q,
                        const void* kv, const int32_t* bt, const int32_t* seq_lens,
                        const int32_t* cu_q, int num_seqs, int total_q, int max_q, int max_kv,
                        int hq, int hkv, int d, int num_pages, float scale, int causal,
                        cudaStream_t stream, const Shape& sh, const void* k_new = nullptr,
                        const void* v_new = nullptr, Mode mode = Mode::kBf16,
                        const QuantBufs* qb = nullptr, bool selftest_abort = false) {
  pattn_status s = PATTN_OK;

  Workspace ws{};
  ws.hdr = reinterpret_cast<int*>(wsb + L.hdr);
  ws.seq_info = reinterpret_cast<int4*>(wsb + L.seq_info);
  ws.seq_plan = reinterpret_cast<int4*>(wsb + L.seq_plan);
  ws.seq_part = reinterpret_cast<int*>(wsb + L.seq_part);
  ws.items = reinterpret_cast<int4*>(wsb + L.items);
  ws.dec_items = reinterpret_cast<int4*>(wsb + L.dec_items);
  ws.unit_cnt = reinterpret_cast<int*>(wsb + L.unit_cnt);
  ws.part_ml = reinterpret_cast<float2*>(wsb + L.part_ml);
  ws.part_o = reinterpret_cast<float*>(wsb + L.part_o);
  ws.max_items = L.max_items;
  ws.max_units = L.max_units;
  ws.max_part_rows = L.max_part_rows;

  // ---- tensor maps (bf16, 128-byte swizzle, 64-element inner boxes)
  const int g = sh.group, T = sh.tokens_per_tile;
  // Units of at most kDecRows packed rows go to the decode kernel, unless the
  // bounds leave no room for one: every sequence holds at least
  // total_q - (num_seqs - 1) * max_q queries. Then the decode kernel is not
  // launched, and the plan sends every unit to the prefill kernel (which serves
  // any unit; a caller whose cu_q ends short of total_q only loses speed).
  const long long min_ql =
      static_cast<long long>(total_q) - static_cast<long long>(num_seqs - 1) * std::max(max_q, 0);
  const bool dec_enabled = g <= kDecRows && min_ql * g <= kDecRows;
  const bool run_prefill = !dec_enabled || static_cast<long long>(max_q) * g > kDecRows;
  CUtensorMap tq{}, tq_dec{}, tkv{}, to{};
  if (mode != Mode::kPlanOnly && dec_enabled) {
    // decode items: the G heads of one KV head for kDecRows / G tokens
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(g),
                                static_cast<cuuint64_t>(hkv),
                                static_cast<cuuint64_t>(std::max(total_q, 1))};
    const cuuint64_t str[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(g) * d * 2,
                               static_cast<cuuint64_t>(hq) * d * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(g), 1,
                               static_cast<cuuint32_t>(kDecRows / g)};
    if ((s = encode(&tq_dec, q, 4, dims, str, box)) != PATTN_OK) return s;
  }
  if (mode != Mode::kPlanOnly) {
    {
      const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(g),
                                  static_cast<cuuint64_t>(hkv),
                                  static_cast<cuuint64_t>(std::max(total_q, 1))};
      const cuuint64_t str[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(g) * d * 2,
                                 static_cast<cuuint64_t>(hq) * d * 2};
      const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(g), 1, static_cast<cuuint32_t>(T)};
      if ((s = encode(&tq, q, 4, dims, str, box)) != PATTN_OK) return s;
      to = tq;
      if (d == 128) {
        // the output (q's shape): 32-channel slices of a q tile's rows, stored by
        // the head_dim-128 prefill kernels
        const cuuint32_t obox[4] = {32, static_cast<cuuint32_t>(g), 1, static_cast<cuuint32_t>(T)};
        if ((s = encode(&to, out, 4, dims, str, obox, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        CU_TENSOR_MAP_SWIZZLE_64B)) != PATTN_OK)
          return s;
      }
    }
    if (bt) {
      const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(kPage),
                                  static_cast<cuuint64_t>(hkv),
                                  static_cast<cuuint64_t>(num_pages) * 2};
      const cuuint64_t str[3] = {static_cast<cuuint64_t>(hkv) * d * 2,
                                 static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(kPage) * hkv * d * 2};
      const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kPage), 1, 1};
      if ((s = encode(&tkv, kv, 4, dims, str, box)) != PATTN_OK) return s;
    } else {
      const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv),
                                  static_cast<cuuint64_t>(num_pages), 2};
      const cuuint64_t str[3] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(hkv) * d * 2,
                                 static_cast<cuuint64_t>(num_pages) * hkv * d * 2};
      const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kPage), 1};
      if ((s = encode(&tkv, kv, 4, dims, str, box)) != PATTN_OK) return s;
    }
  }

  PlanParams pp{};
  pp.cu_q = cu_q;
  pp.seq_lens = seq_lens;
  pp.block_table = bt;
  pp.out = static_cast<__nv_bfloat16*>(out);
  pp.ws = ws;
  pp.num_seqs = num_seqs;
  pp.total_q = total_q;
  pp.max_q = max_q;
  pp.max_kv = max_kv;
  pp.n_heads_q = hq;
  pp.n_heads_kv = hkv;
  pp.group = g;
  pp.head_dim = d;
  pp.tokens_per_tile = T;
  pp.block_n = sh.block_n;
  pp.block_n_shift = sh.block_n == 128 ? 7 : 6;
  // items of two q tiles: the CTA-pair kernel (head_dim 256) and the two-q-tile
  // kernel (head_dim 128, bf16; the quantised modes keep one q tile per item)
  const bool two_q = sh.two_q && (mode == Mode::kBf16 || mode == Mode::kPlanOnly);
  pp.pair = (sh.pair || two_q) ? 1 : 0;
  pp.bt_stride = std::max(1, cdiv(max_kv, kPage));
  pp.num_pages = num_pages;
  pp.causal = causal;
  pp.dec_enabled = dec_enabled ? 1 : 0;
  pp.target_items = plan_target(st.sms);
  pp.min_chunk = kMinChunk;
  pp.ctas = st.sms;
  if (k_new && mode != Mode::kPlanOnly) {
    // the new tokens' K and V rows go into their cache slots from the plan
    // grid's extra CTAs (a warp per token, at most two CTAs per SM), before any
    // attention kernel reads the cache: those wait for the whole plan grid
    pp.k_new = static_cast<const __nv_bfloat16*>(k_new);
    pp.v_new = static_cast<const __nv_bfloat16*>(v_new);
    pp.kv_pool = static_cast<__nv_bfloat16*>(const_cast<void*>(kv));
    pp.write_ctas = std::min(cdiv(total_q, kPlanWarps), 2 * st.sms);
  }

  AttnParams ap{};
  ap.items = ws.items;
  ap.hdr = ws.hdr;
  ap.seq_info = ws.seq_info;
  ap.seq_plan = ws.seq_plan;
  ap.unit_cnt = ws.unit_cnt;
  ap.block_table = bt;
  ap.out = static_cast<__nv_bfloat16*>(out);
  ap.part_o = ws.part_o;
  ap.part_ml = ws.part_ml;
  ap.err = ws.hdr + kHdrErr;
  ap.go = ws.hdr + kHdrGo;
  // bf16 calls that launch both attention kernels: the prefill kernel starts on
  // the decode kernel's go word (the quantised modes' prefill kernel also reads
  // what the quantisation kernels write, so it keeps its grid wait)
  ap.early_start = (mode == Mode::kBf16 && dec_enabled && run_prefill) ? 1 : 0;
  ap.bt_stride = pp.bt_stride;
  ap.num_pages = num_pages;
  ap.n_heads_q = hq;
  ap.n_heads_kv = hkv;
  ap.group = g;
  ap.tokens_per_tile = T;
  ap.scale_log2 = scale * 1.4426950408889634f;
  ap.causal = causal;
  ap.paged = bt ? 1 : 0;
  ap.selftest_abort = selftest_abort ? 1 : 0;

  AttnParams dp = ap;
  dp.items = ws.dec_items;
  dp.tokens_per_tile = dec_enabled ? kDecRows / g : 0;

  const bool prof = g_profile && mode != Mode::kPlanOnly && st.prof.size() < static_cast<size_t>(kProfileCap);
  ProfileRec rec{};
  if (prof) {
    rec = take_events(st);
    cudaEventRecord(rec.ev[0], stream);
  }
  // Every kernel is a dependent launch: it may become resident while its
  // predecessor in the stream finishes, and waits for it on the device before
  // reading anything (the plan rewrites the workspace that the previous call's
  // kernels read, so it too waits for the whole previous grid). Profiling
  // events between the launches turn that overlap off.
  const bool dep = !prof;
  cudaError_t e = cudaSuccess;
  if (mode != Mode::kBf16 && mode != Mode::kPlanOnly) {
    // the key sums of the quantisation start from zero
    e = cudaMemsetAsync(qb->scratch, 0, quant_zero_bytes(num_seqs, hkv, d), stream);
    if (e != cudaSuccess) return PATTN_ERR_CUDA;
  }
  e = launch_plan(pp, stream, dep);
  if (e != cudaSuccess) return PATTN_ERR_CUDA;
  if (mode == Mode::kPlanOnly) return PATTN_OK;
  if (prof) cudaEventRecord(rec.ev[1], stream);
  if (mode != Mode::kBf16) {
    // e4m3 codes and scales of Q, of the smoothed K and of V (dependent launches)
    QuantParams qp{};
    qp.q = static_cast<const __nv_bfloat16*>(q);
    qp.kv_pool = static_cast<const __nv_bfloat16*>(kv);
    qp.block_table = bt;
    qp.seq_info = ws.seq_info;
    qp.q8 = qb->q8;
    qp.q_scale = qb->q_scale;
    qp.k8 = qb->k8;
    qp.k_scale = qb->k_scale;
    qp.v8 = qb->v8;
    qp.v_scale = qb->v_scale;
    qp.sc = quant_scratch_split(qb->scratch, num_seqs, hkv, d);
    qp.num_seqs = num_seqs;
    qp.total_q = total_q;
    qp.n_heads_q = hq;
    qp.n_heads_kv = hkv;
    qp.head_dim = d;
    qp.bt_stride = pp.bt_stride;
    qp.num_pages = num_pages;
    qp.nb_max = qb->nb_max;
    e = launch_quant(qp, st.sms, stream);
    if (e != cudaSuccess) return PATTN_ERR_CUDA;
  }
  if (prof) cudaEventRecord(rec.ev[2], stream);
  if (mode == Mode::kQuantOnly) {
    if (prof) {
      for (int k = 3; k < 6; ++k) cudaEventRecord(rec.ev[k], stream);
      st.prof.push_back(rec);
    }
    return PATTN_OK;
  }
  if (dec_enabled) {
    e = launch_decode(dp, tq_dec, tkv, d, st.sms, stream, dep);
    if (e != cudaSuccess) return PATTN_ERR_CUDA;
  }
  if (prof) cudaEventRecord(rec.ev[3], stream);
  if (run_prefill) {
    if (mode == Mode::kFp8 || mode == Mode::kFp8Pv) {
      // e4m3 Q [total_q][hq][d] and K blocks [B * nb_max][64][hkv][d], one byte each
      CUtensorMap tq8, tk8;
      const cuuint64_t qdims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(g),
                                   static_cast<cuuint64_t>(hkv),
                                   static_cast<cuuint64_t>(std::max(total_q, 1))};
      const cuuint64_t qstr[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(g) * d,
                                  static_cast<cuuint64_t>(hq) * d};
      const cuuint32_t qbox[4] = {128, static_cast<cuuint32_t>(g), 1, static_cast<cuuint32_t>(T)};
      if ((s = encode(&tq8, qb->q8, 4, qdims, qstr, qbox, CU_TENSOR_MAP_DATA_TYPE_UINT8)) != PATTN_OK)
        return s;
      const cuuint64_t kdims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(kPage),
                                   static_cast<cuuint64_t>(hkv),
                                   static_cast<cuuint64_t>(num_seqs) * qb->nb_max};
      const cuuint64_t kstr[3] = {static_cast<cuuint64_t>(hkv) * d, static_cast<cuuint64_t>(d),
                                  static_cast<cuuint64_t>(kPage) * hkv * d};
      const cuuint32_t kbox[4] = {128, static_cast<cuuint32_t>(kPage), 1, 1};
      if ((s = encode(&tk8, qb->k8, 4, kdims, kstr, kbox, CU_TENSOR_MAP_DATA_TYPE_UINT8)) != PATTN_OK)
        return s;
      AttnParams fp = ap;
      fp.q_scale = qb->q_scale;
      fp.k_scale = qb->k_scale;
      fp.nb_max = qb->nb_max;
      if (mode == Mode::kFp8Pv) {
        // transposed e4m3 V tiles [B * nb_max / 2][hkv][d][128 keys]
        CUtensorMap tv8;
        const cuuint64_t vdims[4] = {128, static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv),
                                     static_cast<cuuint64_t>(num_seqs) * (qb->nb_max / 2)};
        const cuuint64_t vstr[3] = {128, static_cast<cuuint64_t>(d) * 128,
                                    static_cast<cuuint64_t>(hkv) * d * 128};
        const cuuint32_t vbox[4] = {128, static_cast<cuuint32_t>(d), 1, 1};
        if ((s = encode(&tv8, qb->v8, 4, vdims, vstr, vbox, CU_TENSOR_MAP_DATA_TYPE_UINT8)) != PATTN_OK)
          return s;
        fp.v_scale = qb->v_scale;
        e = launch_attention_fp8pv(fp, tq8, tk8, tv8, to, st.sms, stream, dep);
      } else {
        e = launch_attention_fp8(fp, tq8, tk8, tkv, to, st.sms, stream, dep);
      }
    } else {
      e = sh.pair   ? launch_attention_pair(ap, tq, tkv, st.sms, stream, dep)
          : two_q   ? launch_attention_2q(ap, tq, tkv, to, st.sms, stream, dep)
                    : launch_attention(ap, tq, tkv, to, d, st.sms, stream, dep);
    }
    if (e != cudaSuccess) return PATTN_ERR_CUDA;
  }
  if (prof) cudaEventRecord(rec.ev[4], stream);
  // (split units are merged inside the attention kernels, by the CTA that
  // finishes a unit's last split)
  if (prof) {
    cudaEventRecord(rec.ev[5], stream);
    st.prof.push_back(rec);
  }
  return PATTN_OK;
}

pattn_status forward_locked(void* out, const void* q, const void* kv, const int32_t* bt,
                            const int32_t* seq_lens, const int32_t* cu_q, int num_seqs,
                            int total_q, int max_q, int max_kv, int hq, int hkv, int d, int page,
                            int num_pages, float scale, int causal, cudaStream_t stream,
                            const Shape& sh, const void* k_new = nullptr,
                            const void* v_new = nullptr, Mode mode = Mode::kBf16,
                            bool selftest_abort = false) {
  (void)page;
  DeviceState* stp = nullptr;
  pattn_status s = device_state(&stp);
  if (s != PATTN_OK) return s;
  DeviceState& st = *stp;
  const WsLayout L = ws_layout(num_seqs, total_q, max_q, hq, hkv, d);
  const Fp8Layout F = fp8_layout(L.total, num_seqs, total_q, max_kv, hq, hkv, d, mode == Mode::kFp8Pv);
  const bool quant = mode != Mode::kBf16 && mode != Mode::kPlanOnly;
  if ((s = ensure_workspace(st, quant ? F.total : L.total)) != PATTN_OK) return s;
  uint8_t* wsb = static_cast<uint8_t*>(st.ws);
  QuantBufs qb;
  if (quant) {
    qb.q8 = wsb + F.q8;
    qb.q_scale = reinterpret_cast<float*>(wsb + F.q_scale);
    qb.k8 = wsb + F.k8;
    qb.k_scale = reinterpret_cast<float*>(wsb + F.k_scale);
    qb.scratch = wsb + F.k_sum;
    qb.nb_max = F.nb_max;
    if (mode == Mode::kFp8Pv) {
      qb.v8 = wsb + F.v8;
      qb.v_scale = reinterpret_cast<float*>(wsb + F.v_scale);
    }
  }
  return launch_all(st, wsb, L, out, q, kv, bt, seq_lens, cu_q, num_seqs, total_q, max_q, max_kv, hq,
                    hkv, d, num_pages, scale, causal, stream, sh, k_new, v_new, mode, &qb, selftest_abort);
}

// ---------------------------------------------------------------------------
// Fixed scratch for pattn_forward_noalloc: one file-scope device array that
// every GPU loading the library holds until the process exits. Host code only
// sees a stand-in symbol; the device address comes from cudaGetSymbolAddress,
// taken once per device at set-up with that device current.
static __device__ __align__(256) uint8_t g_noalloc_scratch[PATTN_NOALLOC_SCRATCH_BYTES];
uint8_t* g_noalloc_ptr[kMaxDevices] = {};

// Caller holds g_mu; `dev` is the current device.
pattn_status noalloc_scratch(int dev, uint8_t** out) {
  if (dev < 0 || dev >= kMaxDevices) return PATTN_ERR_UNSUPPORTED;
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return PATTN_ERR_CUDA;
    // the device error word and counters of the header start at zero
    if (cudaMemset(ptr, 0, kHdrWords * sizeof(int)) != cudaSuccess) return PATTN_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return PATTN_OK;
}

}  // namespace
}  // namespace pattn

using namespace pattn;

extern "C" {

pattn_status pattn_forward(void* out, const void* q, const void* kv_pool,
                           const int32_t* block_table, const int32_t* seq_lens,
                           const int32_t* cu_q, int num_seqs, int total_q, int max_q, int max_kv,
                           int n_heads_q, int n_heads_kv, int head_dim, int page_size,
                           int num_pages, float scale, int causal, pattn_stream_t stream) {
  Shape sh{};
  pattn_status s = check_args(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q,
                              max_q, max_kv, n_heads_q, n_heads_kv, head_dim, page_size,
                              num_pages, scale, causal, &sh);
  if (s != PATTN_OK) return s;
  if (num_seqs == 0 || total_q == 0) return PATTN_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  return forward_locked(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q, max_q,
                        max_kv, n_heads_q, n_heads_kv, head_dim, page_size, num_pages, scale,
                        causal, reinterpret_cast<cudaStream_t>(stream), sh);
}

pattn_status pattn_forward_append(void* out, const void* q, const void* k_new, const void* v_new,
                                  void* kv_pool, const int32_t* block_table,
                                  const int32_t* seq_lens, const int32_t* cu_q, int num_seqs,
                                  int total_q, int max_q, int max_kv, int n_heads_q,
                                  int n_heads_kv, int head_dim, int page_size, int num_pages,
                                  float scale, int causal, pattn_stream_t stream) {
  Shape sh{};
  pattn_status s = check_args(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q,
                              max_q, max_kv, n_heads_q, n_heads_kv, head_dim, page_size,
                              num_pages, scale, causal, &sh);
  if (s != PATTN_OK) return s;
  if (total_q > 0 && (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)))
    return PATTN_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0) return PATTN_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  return forward_locked(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q, max_q,
                        max_kv, n_heads_q, n_heads_kv, head_dim, page_size, num_pages, scale,
                        causal, reinterpret_cast<cudaStream_t>(stream), sh, k_new, v_new);
}

pattn_status pattn_forward_fp8qk(void* out, const void* q, const void* kv_pool,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 const int32_t* cu_q, int num_seqs, int total_q, int max_q, int max_kv,
                                 int n_heads_q, int n_heads_kv, int head_dim, int page_size,
                                 int num_pages, float scale, int causal, pattn_stream_t stream) {
  Shape sh{};
  pattn_status s = check_args(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q,
                              max_q, max_kv, n_heads_q, n_heads_kv, head_dim, page_size,
                              num_pages, scale, causal, &sh);
  if (s != PATTN_OK) return s;
  if (head_dim != 128 || max_kv > kFp8MaxKv) return PATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_seqs) * n_heads_kv > 0x7fffffffLL) return PATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0) return PATTN_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  return forward_locked(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q, max_q,
                        max_kv, n_heads_q, n_heads_kv, head_dim, page_size, num_pages, scale,
                        causal, reinterpret_cast<cudaStream_t>(stream), sh, nullptr, nullptr,
                        Mode::kFp8);
}

pattn_status pattn_forward_fp8(void* out, const void* q, const void* kv_pool, const int32_t* block_table,
                               const int32_t* seq_lens, const int32_t* cu_q, int num_seqs, int total_q,
                               int max_q, int max_kv, int n_heads_q, int n_heads_kv, int head_dim,
                               int page_size, int num_pages, float scale, int causal, pattn_stream_t stream) {
  Shape sh{};
  pattn_status s = check_args(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q,
                              max_q, max_kv, n_heads_q, n_heads_kv, head_dim, page_size,
                              num_pages, scale, causal, &sh);
  if (s != PATTN_OK) return s;
  if (head_dim != 128 || max_kv > kFp8MaxKv) return PATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_seqs) * n_heads_kv > 0x7fffffffLL) return PATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0) return PATTN_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  return forward_locked(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q, max_q,
                        max_kv, n_heads_q, n_heads_kv, head_dim, page_size, num_pages, scale,
                        causal, reinterpret_cast<cudaStream_t>(stream), sh, nullptr, nullptr,
                        Mode::kFp8Pv);
}

pattn_status pattn_quantize_qk(void* q8, float* q_scale, void* k8, float* k_scale, const void* q,
                               const void* kv_pool, const int32_t* block_table,
                               const int32_t* seq_lens, const int32_t* cu_q, int num_seqs,
                               int total_q, int max_q, int max_kv, int n_heads_q, int n_heads_kv,
                               int head_dim, int page_size, int num_pages, pattn_stream_t stream) {
  Shape sh{};
  // the attention's argument rules (a dummy output pointer; scale and causal unused)
  pattn_status s = check_args(q, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q, max_q,
                              max_kv, n_heads_q, n_heads_kv, head_dim, page_size, num_pages, 1.0f, 0,
                              &sh);
  if (s != PATTN_OK) return s;
  if (!q8 || !q_scale || !k8 || !k_scale || !aligned(q8, 16) || !aligned(k8, 16) ||
      !aligned(q_scale, 4) || !aligned(k_scale, 4))
    return PATTN_ERR_INVALID_ARG;
  if (head_dim != 128 || max_kv > kFp8MaxKv) return PATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0) return PATTN_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* stp = nullptr;
  if ((s = device_state(&stp)) != PATTN_OK) return s;
  DeviceState& st = *stp;
  const WsLayout L = ws_layout(num_seqs, total_q, max_q, n_heads_q, n_heads_kv, head_dim);
  const Fp8Layout F = fp8_layout(L.total, num_seqs, total_q, max_kv, n_heads_q, n_heads_kv, head_dim);
  const size_t need = align_up(F.k_sum + quant_scratch_bytes(num_seqs, n_heads_kv, head_dim), 256);
  if ((s = ensure_workspace(st, need)) != PATTN_OK) return s;
  uint8_t* wsb = static_cast<uint8_t*>(st.ws);
  QuantBufs qb;
  qb.q8 = static_cast<uint8_t*>(q8);
  qb.q_scale = q_scale;
  qb.k8 = static_cast<uint8_t*>(k8);
  qb.k_scale = k_scale;
  qb.scratch = wsb + F.k_sum;
  qb.nb_max = F.nb_max;
  return launch_all(st, wsb, L, nullptr, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q,
                    max_q, max_kv, n_heads_q, n_heads_kv, head_dim, num_pages, 1.0f, 0,
                    reinterpret_cast<cudaStream_t>(stream), sh, nullptr, nullptr, Mode::kQuantOnly,
                    &qb);
}

pattn_status pattn_quantize_v(void* v8, float* v_scale, const void* kv_pool, const int32_t* block_table,
                              const int32_t* seq_lens, const int32_t* cu_q, int num_seqs, int total_q,
                              int max_q, int max_kv, int n_heads_q, int n_heads_kv, int head_dim,
                              int page_size, int num_pages, pattn_stream_t stream) {
  Shape sh{};
  // the attention's argument rules (dummy output and query pointers: neither is read)
  pattn_status s = check_args(kv_pool, kv_pool, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q,
                              max_q, max_kv, n_heads_q, n_heads_kv, head_dim, page_size, num_pages, 1.0f,
                              0, &sh);
  if (s != PATTN_OK) return s;
  if (!v8 || !v_scale || !aligned(v8, 16) || !aligned(v_scale, 16)) return PATTN_ERR_INVALID_ARG;
  if (head_dim != 128 || max_kv > kFp8MaxKv) return PATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0) return PATTN_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* stp = nullptr;
  if ((s = device_state(&stp)) != PATTN_OK) return s;
  DeviceState& st = *stp;
  const WsLayout L = ws_layout(num_seqs, total_q, max_q, n_heads_q, n_heads_kv, head_dim);
  const Fp8Layout F = fp8_layout(L.total, num_seqs, total_q, max_kv, n_heads_q, n_heads_kv, head_dim);
  const size_t need = align_up(F.k_sum + quant_scratch_bytes(num_seqs, n_heads_kv, head_dim), 256);
  if ((s = ensure_workspace(st, need)) != PATTN_OK) return s;
  uint8_t* wsb = static_cast<uint8_t*>(st.ws);
  QuantBufs qb;
  qb.v8 = static_cast<uint8_t*>(v8);
  qb.v_scale = v_scale;
  qb.scratch = wsb + F.k_sum;
  qb.nb_max = F.nb_max;
  return launch_all(st, wsb, L, nullptr, kv_pool, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q,
                    max_q, max_kv, n_heads_q, n_heads_kv, head_dim, num_pages, 1.0f, 0,
                    reinterpret_cast<cudaStream_t>(stream), sh, nullptr, nullptr, Mode::kQuantOnly, &qb);
}

size_t pattn_workspace_size_fp8(int num_seqs, int total_q, int max_q, int max_kv, int n_heads_q,
                                int n_heads_kv, int head_dim, int page_size) {
  (void)page_size;
  if (num_seqs < 0 || total_q < 0 || max_q < 0 || max_kv < 0 || n_heads_q <= 0 || n_heads_kv <= 0 ||
      n_heads_q % n_heads_kv != 0 || n_heads_q / n_heads_kv > kBM || head_dim != 128 ||
      max_kv > kFp8MaxKv)
    return 0;
  const WsLayout L = ws_layout(num_seqs, total_q, max_q, n_heads_q, n_heads_kv, head_dim);
  return fp8_layout(L.total, num_seqs, total_q, max_kv, n_heads_q, n_heads_kv, head_dim, true).total;
}

size_t pattn_workspace_size_fp8qk(int num_seqs, int total_q, int max_q, int max_kv, int n_heads_q,
                                  int n_heads_kv, int head_dim, int page_size) {
  (void)page_size;
  if (num_seqs < 0 || total_q < 0 || max_q < 0 || max_kv < 0 || n_heads_q <= 0 || n_heads_kv <= 0 ||
      n_heads_q % n_heads_kv != 0 || n_heads_q / n_heads_kv > kBM || head_dim != 128 ||
      max_kv > kFp8MaxKv)
    return 0;
  const WsLayout L = ws_layout(num_seqs, total_q, max_q, n_heads_q, n_heads_kv, head_dim);
  return fp8_layout(L.total, num_seqs, total_q, max_kv, n_heads_q, n_heads_kv, head_dim).total;
}

pattn_status pattn_forward_noalloc(void* out, const void* q, const void* kv_pool,
                                   const int32_t* block_table, const int32_t* seq_lens,
                                   const int32_t* cu_q, int num_seqs, int total_q, int max_q,
                                   int max_kv, int n_heads_q, int n_heads_kv, int head_dim,
                                   int page_size, int num_pages, float scale, int causal,
                                   pattn_stream_t stream) {
  Shape sh{};
  pattn_status s = check_args(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q,
                              max_q, max_kv, n_heads_q, n_heads_kv, head_dim, page_size,
                              num_pages, scale, causal, &sh);
  if (s != PATTN_OK) return s;
  if (num_seqs == 0 || total_q == 0) return PATTN_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* stp = nullptr;
  if ((s = device_state(&stp)) != PATTN_OK) return s;
  const WsLayout L = ws_layout(num_seqs, total_q, max_q, n_heads_q, n_heads_kv, head_dim, max_kv,
                              plan_target_max(stp->sms));
  if (L.total > static_cast<size_t>(PATTN_NOALLOC_SCRATCH_BYTES)) return PATTN_ERR_NO_MEMORY;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PATTN_ERR_CUDA;
  uint8_t* scratch = nullptr;
  if ((s = noalloc_scratch(dev, &scratch)) != PATTN_OK) return s;
  return launch_all(*stp, scratch, L, out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs,
                    total_q, max_q, max_kv, n_heads_q, n_heads_kv, head_dim, num_pages, scale,
                    causal, reinterpret_cast<cudaStream_t>(stream), sh);
}

pattn_status pattn_forward_host(void* out, const void* q, const void* kv_pool,
                                size_t kv_pool_bytes, const int32_t* block_table,
                                const int32_t* seq_lens, const int32_t* cu_q, int num_seqs,
                                int total_q, int max_q, int max_kv, int n_heads_q, int n_heads_kv,
                                int head_dim, int page_size, int num_pages, float scale,
                                int causal, pattn_stream_t stream) {
  Shape sh{};
  pattn_status s = check_args(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q,
                              max_q, max_kv, n_heads_q, n_heads_kv, head_dim, page_size,
                              num_pages, scale, causal, &sh);
  if (s != PATTN_OK) return s;
  if (kv_pool_bytes == 0) return PATTN_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0) return PATTN_OK;
  cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* stp = nullptr;
  if ((s = device_state(&stp)) != PATTN_OK) return s;
  DeviceState& st = *stp;
  const size_t qo_bytes = static_cast<size_t>(total_q) * n_heads_q * head_dim * 2;
  const size_t bt_bytes =
      block_table ? static_cast<size_t>(num_seqs) * std::max(1, cdiv(max_kv, page_size)) * 4 : 0;
  const size_t need[6] = {qo_bytes, kv_pool_bytes, std::max<size_t>(bt_bytes, 16),
                          static_cast<size_t>(num_seqs) * 4, static_cast<size_t>(num_seqs + 1) * 4,
                          qo_bytes};
  for (int i = 0; i < 6; ++i) {
    if (st.stage[i] && st.stage_bytes[i] >= need[i]) continue;
    if (st.stage[i]) {
      cudaDeviceSynchronize();
      cudaFree(st.stage[i]);
      st.stage[i] = nullptr;
      st.stage_bytes[i] = 0;
    }
    cudaError_t e = cudaMalloc(&st.stage[i], need[i]);
    if (e != cudaSuccess) {
      st.stage[i] = nullptr;
      return cuda_fail(e);
    }
    st.stage_bytes[i] = need[i];
  }
  cudaError_t e = cudaSuccess;
  const void* src[5] = {q, kv_pool, block_table, seq_lens, cu_q};
  const size_t n[5] = {qo_bytes, kv_pool_bytes, bt_bytes, static_cast<size_t>(num_seqs) * 4,
                       static_cast<size_t>(num_seqs + 1) * 4};
  for (int i = 0; i < 5 && e == cudaSuccess; ++i)
    if (src[i] && n[i]) e = cudaMemcpyAsync(st.stage[i], src[i], n[i], cudaMemcpyHostToDevice, st_);
  if (e != cudaSuccess) return PATTN_ERR_CUDA;
  s = forward_locked(st.stage[5], st.stage[0], st.stage[1],
                     block_table ? static_cast<const int32_t*>(st.stage[2]) : nullptr,
                     static_cast<const int32_t*>(st.stage[3]), static_cast<const int32_t*>(st.stage[4]),
                     num_seqs, total_q, max_q, max_kv, n_heads_q, n_heads_kv, head_dim, page_size,
                     num_pages, scale, causal, st_, sh);
  if (s != PATTN_OK) return s;
  e = cudaMemcpyAsync(out, st.stage[5], qo_bytes, cudaMemcpyDeviceToHost, st_);
  if (e != cudaSuccess) return PATTN_ERR_CUDA;
  e = cudaStreamSynchronize(st_);
  return e == cudaSuccess ? PATTN_OK : PATTN_ERR_CUDA;
}

size_t pattn_workspace_size(int num_seqs, int total_q, int max_q, int max_kv, int n_heads_q,
                            int n_heads_kv, int head_dim, int page_size) {
  (void)max_kv;
  (void)page_size;
  if (num_seqs < 0 || total_q < 0 || max_q < 0 || n_heads_q <= 0 || n_heads_kv <= 0 ||
      n_heads_q % n_heads_kv != 0 || n_heads_q / n_heads_kv > kBM || (head_dim != 128 && head_dim != 256))
    return 0;
  return ws_layout(num_seqs, total_q, max_q, n_heads_q, n_heads_kv, head_dim).total;
}

pattn_status pattn_set_workspace(void* ptr, size_t bytes) {
  if (ptr && (!aligned(ptr, 256) || bytes < kHdrWords * sizeof(int))) return PATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* stp = nullptr;
  pattn_status s = device_state(&stp);
  if (s != PATTN_OK) return s;
  DeviceState& st = *stp;
  if (!st.ws_caller && st.ws) {
    cudaDeviceSynchronize();
    cudaFree(st.ws);
  }
  st.ws = nullptr;
  st.ws_bytes = 0;
  st.ws_caller = false;
  if (ptr) {
    if (cudaMemset(ptr, 0, kHdrWords * sizeof(int)) != cudaSuccess) return PATTN_ERR_CUDA;
    st.ws = ptr;
    st.ws_bytes = bytes;
    st.ws_caller = true;
  }
  return PATTN_OK;
}

pattn_status pattn_get_device_status(pattn_stream_t stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* stp = nullptr;
  pattn_status s = device_state(&stp);
  if (s != PATTN_OK) return s;
  cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st_) != cudaSuccess) return PATTN_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PATTN_ERR_CUDA;
  // the error words of the library (or caller) workspace and of the fixed
  // scratch behind pattn_forward_noalloc, each read and cleared (no allocation)
  void* words[2] = {stp->ws, g_noalloc_ptr[dev]};
  int err = 0;
  for (void* w : words) {
    if (!w) continue;
    int e = 0;
    if (cudaMemcpy(&e, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PATTN_ERR_CUDA;
    if (e && cudaMemset(w, 0, sizeof(int)) != cudaSuccess) return PATTN_ERR_CUDA;
    err |= e;
  }
  if (err & kErrTimeout) return PATTN_ERR_DEVICE_TIMEOUT;
  if (err & kErrBadInput) return PATTN_ERR_DEVICE_BAD_INPUT;
  return PATTN_OK;
}

pattn_status pattn_selftest_wait_timeout(pattn_stream_t stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* stp = nullptr;
  pattn_status s = device_state(&stp);
  if (s != PATTN_OK) return s;
  if ((s = ensure_workspace(*stp, kHdrWords * sizeof(int))) != PATTN_OK) return s;
  const cudaError_t e = launch_wait_selftest(static_cast<int*>(stp->ws), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PATTN_OK : PATTN_ERR_CUDA;
}

pattn_status pattn_selftest_attention_timeout(void* out, const void* q, const void* kv_pool,
                                              const int32_t* block_table, const int32_t* seq_lens,
                                              const int32_t* cu_q, int num_seqs, int total_q, int max_q,
                                              int max_kv, int n_heads_q, int n_heads_kv, int head_dim,
                                              int page_size, int num_pages, float scale, int causal,
                                              pattn_stream_t stream) {
  Shape sh{};
  pattn_status s = check_args(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q,
                              max_q, max_kv, n_heads_q, n_heads_kv, head_dim, page_size,
                              num_pages, scale, causal, &sh);
  if (s != PATTN_OK) return s;
  if (sh.pair) return PATTN_ERR_UNSUPPORTED;  // the CTA-pair kernel has no self-test wait
  if (num_seqs == 0 || total_q == 0) return PATTN_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  return forward_locked(out, q, kv_pool, block_table, seq_lens, cu_q, num_seqs, total_q, max_q,
                        max_kv, n_heads_q, n_heads_kv, head_dim, page_size, num_pages, scale,
                        causal, reinterpret_cast<cudaStream_t>(stream), sh, nullptr, nullptr,
                        Mode::kBf16, true);
}

pattn_status pattn_plan_items(const int32_t* block_table, const int32_t* seq_lens, const int32_t* cu_q,
                              int num_seqs, int total_q, int max_q, int max_kv, int n_heads_q,
                              int n_heads_kv, int head_dim, int page_size, int num_pages, int causal,
                              int32_t* prefill_items, int32_t* decode_items, int capacity, int32_t* counts,
                              pattn_stream_t stream) {
  Shape sh{};
  pattn_status s = check_shape(block_table, seq_lens, cu_q, num_seqs, total_q, max_q, max_kv, n_heads_q,
                               n_heads_kv, head_dim, page_size, num_pages, 1.0f, causal, &sh);
  if (s != PATTN_OK) return s;
  if (!counts || capacity < 0 || (capacity > 0 && (!prefill_items || !decode_items))) return PATTN_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) counts[i] = 0;
  if (num_seqs == 0 || total_q == 0) return PATTN_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if ((s = forward_locked(nullptr, nullptr, nullptr, block_table, seq_lens, cu_q, num_seqs, total_q, max_q,
                          max_kv, n_heads_q, n_heads_kv, head_dim, page_size, num_pages, 1.0f, causal, cs, sh,
                          nullptr, nullptr, Mode::kPlanOnly)) != PATTN_OK)
    return s;
  DeviceState* stp = nullptr;
  if ((s = device_state(&stp)) != PATTN_OK) return s;
  const WsLayout L = ws_layout(num_seqs, total_q, max_q, n_heads_q, n_heads_kv, head_dim);
  const uint8_t* wsb = static_cast<const uint8_t*>(stp->ws);
  int hdr[kHdrWords];
  if (cudaMemcpyAsync(hdr, wsb + L.hdr, sizeof(hdr), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
      cudaStreamSynchronize(cs) != cudaSuccess)
    return PATTN_ERR_CUDA;
  counts[0] = hdr[kHdrItems];
  counts[1] = hdr[kHdrDecItems];
  counts[2] = hdr[kHdrUnits];
  counts[3] = hdr[kHdrPartRows];
  const size_t n0 = static_cast<size_t>(std::min(std::max(hdr[kHdrItems], 0), capacity));
  const size_t n1 = static_cast<size_t>(std::min(std::max(hdr[kHdrDecItems], 0), capacity));
  if ((n0 && cudaMemcpyAsync(prefill_items, wsb + L.items, n0 * sizeof(int4), cudaMemcpyDeviceToHost, cs) !=
                 cudaSuccess) ||
      (n1 && cudaMemcpyAsync(decode_items, wsb + L.dec_items, n1 * sizeof(int4), cudaMemcpyDeviceToHost, cs) !=
                 cudaSuccess) ||
      cudaStreamSynchronize(cs) != cudaSuccess)
    return PATTN_ERR_CUDA;
  return hdr[kHdrOverflow] ? PATTN_ERR_NO_MEMORY : PATTN_OK;
}

const char* pattn_status_string(pattn_status status) {
  switch (status) {
    case PATTN_OK: return "ok";
    case PATTN_ERR_INVALID_ARG: return "invalid argument";
    case PATTN_ERR_UNSUPPORTED: return "unsupported shape or device";
    case PATTN_ERR_CUDA: return "CUDA call failed";
    case PATTN_ERR_NO_MEMORY: return "out of device memory or workspace too small";
    case PATTN_ERR_DEVICE_BAD_INPUT: return "device data rejected (page index, lengths or cu_q)";
    case PATTN_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
  }
  return "unknown status";
}

pattn_status pattn_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_profile = on != 0;
  return PATTN_OK;
}

// Sums the recorded calls' per-kernel device time: plan, cache write, decode
// kernel, prefill kernel, after the attention kernels. Caller holds g_mu.
pattn_status profile_sum(double t[5], int* calls) {
  DeviceState* stp = nullptr;
  pattn_status s = device_state(&stp);
  if (s != PATTN_OK) return s;
  DeviceState& st = *stp;
  for (int k = 0; k < 5; ++k) t[k] = 0.0;
  for (auto& r : st.prof) {
    if (cudaEventSynchronize(r.ev[5]) != cudaSuccess) return PATTN_ERR_CUDA;
    for (int k = 0; k < 5; ++k) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, r.ev[k], r.ev[k + 1]) != cudaSuccess) return PATTN_ERR_CUDA;
      t[k] += ms;
    }
  }
  if (calls) *calls = static_cast<int>(st.prof.size());
  for (auto& r : st.prof) st.prof_pool.push_back(r);
  st.prof.clear();
  return PATTN_OK;
}

pattn_status pattn_profile_read(double* ms_plan, double* ms_attention, double* ms_combine,
                                int* calls) {
  std::lock_guard<std::mutex> lk(g_mu);
  double t[5];
  const pattn_status s = profile_sum(t, calls);
  if (s != PATTN_OK) return s;
  if (ms_plan) *ms_plan = t[0];
  if (ms_attention) *ms_attention = t[2] + t[3];
  if (ms_combine) *ms_combine = t[4];
  return PATTN_OK;
}

pattn_status pattn_profile_read_kernels(double* ms, int* calls) {
  if (!ms) return PATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  return profile_sum(ms, calls);
}

}  // extern "C"
