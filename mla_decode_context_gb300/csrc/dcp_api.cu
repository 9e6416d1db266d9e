// C ABI of the DCP MLA hot path: host-side validation, the split-KV plan and
// kernel launches.  No allocation, no synchronisation, no global state.
#include "dcp_kernels.h"

#include <cmath>
#include <cstdint>
#include <cstdlib>

using dcp::DecodeArgs;
using dcp::SplitPlan;

namespace dcp {

namespace {
constexpr int kTargetCtasPerUnit = 2;  // CTAs the decode spends on one (row, shard, split)
constexpr int32_t kMinSplitTokens = 256;
constexpr int32_t kSplitRound = 32;  // split chunks in whole 32-token tiles
constexpr int kMaxSplits = 32;

// CTAs one wave of the decode can hold: the tensor-core kernel's resident
// cluster count x 2 (one CTA per SM), else the SM count, else GB300's 152.
int current_sm_count() {
  const int tc = decode_tc_resident_ctas();
  if (tc > 0) return tc;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();  // clear: no device is not an error for sizing
    return 152;          // GB300
  }
  return sms;
}
}  // namespace

// Most splits a (row, shard) pair with up to `lmax` local tokens may use:
// enough (row, shard, split) units to give every SM work when there are few
// rows (long-context B=1 decode), never splits shorter than kMinSplitTokens.
static int64_t split_cap(int32_t T, int32_t D, int64_t lmax, int sm_count) {
  const int64_t units = static_cast<int64_t>(T) * D * kTargetCtasPerUnit;
  int64_t want = sm_count / units;  // whole waves only
  const int64_t cap_len = (lmax + kMinSplitTokens - 1) / kMinSplitTokens;
  if (want > cap_len) want = cap_len;
  if (want > kMaxSplits) want = kMaxSplits;
  return want < 1 ? 1 : want;
}

// Split-KV plan: pure function of its arguments (and the SM count).
SplitPlan plan_splits(int32_t T, int32_t D, int32_t I, int32_t d0, int32_t Dn, int32_t max_seq_len, int sm_count) {
  SplitPlan p{1, kSplitRound};
  // the first computed shard is the largest of them
  const int32_t lmax = local_len(max_seq_len < 0 ? 0 : max_seq_len, d0, D, I);
  if (lmax <= 0) return p;
  const int64_t want = split_cap(T, Dn, lmax, sm_count);
  int64_t chunk = (lmax + want - 1) / want;
  chunk = (chunk + kSplitRound - 1) / kSplitRound * kSplitRound;
  p.chunk = static_cast<int32_t>(chunk);
  p.splits = static_cast<int32_t>((lmax + chunk - 1) / chunk);  // <= want
  if (p.splits < 1) p.splits = 1;
  return p;
}

// Tail of the workspace for the units' launch order (one int32 per unit).
size_t order_workspace_bytes(const SplitPlan& p, int32_t T, int32_t D) {
  const size_t units = static_cast<size_t>(p.splits < 1 ? 1 : p.splits) * D * T;
  return (units * sizeof(int32_t) + 255) / 256 * 256;
}

size_t split_workspace_bytes(const SplitPlan& p, int32_t T, int32_t H, int32_t D) {
  if (p.splits <= 1) return 0;
  const size_t pairs = static_cast<size_t>(p.splits) * D * T * H;
  size_t bytes = pairs * kLatent * sizeof(float);
  bytes = (bytes + 255) / 256 * 256;
  bytes += pairs * sizeof(float);
  return (bytes + 255) / 256 * 256;
}

}  // namespace dcp

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

namespace {
// What one dcp_mla_decode_partial call with these sizes does on the current
// device: its split plan, the workspace the split partials need, and which
// kernels it launches.
struct DecodeLaunch {
  dcp::SplitPlan plan;
  size_t need;       // split partials (required when plan.splits > 1)
  size_t obytes;     // launch order of the units (optional tail)
  bool simt;         // CUDA-core kernel instead of the tensor-core one
  bool use_order;    // units start longest first (order kernel launched)
};

DecodeLaunch decode_launch(int32_t T, int32_t H, int32_t D, int32_t interleave, int32_t d0, int32_t Dn,
                           int32_t max_seq_len, bool have_workspace, size_t workspace_bytes, bool kv_fp8 = false) {
  DecodeLaunch L{};
  const int sms = dcp::current_sm_count();
  L.plan = dcp::plan_splits(T, D, interleave, d0, Dn, max_seq_len, sms);
  L.need = dcp::split_workspace_bytes(L.plan, T, H, Dn);
  L.obytes = dcp::order_workspace_bytes(L.plan, T, Dn);
  dcp::DecodeArgs a{};
  a.H = H;
  a.plan = L.plan;
  a.kv_fp8 = kv_fp8 ? 1 : 0;
  const char* force = std::getenv("DCP_FORCE_SIMT");  // 1: the CUDA-core reference kernel (A/B checks)
  L.simt = (force && force[0] == '1') || !dcp::decode_tc_supported(a);
  const int64_t units = static_cast<int64_t>(T) * Dn * L.plan.splits;
  const int resident = dcp::decode_tc_resident_ctas();  // 0: no device to size against
  L.use_order = !L.simt && resident > 0 && units > resident / 2 && have_workspace &&
                workspace_bytes >= L.need + L.obytes;
  return L;
}
}  // namespace

extern "C" {

const char* dcp_status_str(dcp_status_t s) {
  switch (s) {
    case DCP_OK: return "DCP_OK";
    case DCP_ERR_INVALID_ARG: return "DCP_ERR_INVALID_ARG";
    case DCP_ERR_UNSUPPORTED_DTYPE: return "DCP_ERR_UNSUPPORTED_DTYPE";
    case DCP_ERR_MISALIGNED: return "DCP_ERR_MISALIGNED";
    case DCP_ERR_TABLE_TOO_NARROW: return "DCP_ERR_TABLE_TOO_NARROW";
    case DCP_ERR_WORKSPACE_TOO_SMALL: return "DCP_ERR_WORKSPACE_TOO_SMALL";
    case DCP_ERR_CUDA: return "DCP_ERR_CUDA";
    case DCP_ERR_TIMEOUT: return "DCP_ERR_TIMEOUT";
  }
  return "DCP_ERR_UNKNOWN";
}

int dcp_version(void) { return 1; }

int32_t dcp_shard_of(int64_t pos, int32_t D, int32_t interleave) {
  if (D < 1 || interleave < 1 || pos < 0) return -1;
  return dcp::shard_of(pos, D, interleave);
}

int32_t dcp_local_len(int32_t L, int32_t d, int32_t D, int32_t interleave) {
  if (L < 0 || D < 1 || interleave < 1 || d < 0 || d >= D) return -1;
  return dcp::local_len(L, d, D, interleave);
}

size_t dcp_decode_workspace_size(int32_t B, int32_t T, int32_t H, int32_t D, int32_t max_seq_len,
                                 int32_t max_q_len) {
  if (B < 0 || T < 0 || H < 1 || D < 1 || D > DCP_MAX_SHARDS || max_seq_len < 0 || max_q_len < 0)
    return static_cast<size_t>(-1);
  if (B == 0 || T == 0) return 0;
  // Upper bound over every interleave: a shard never owns more than
  // max_seq_len tokens, and the split count never exceeds split_cap(lmax).
  const int sms = dcp::current_sm_count();
  dcp::SplitPlan p{static_cast<int32_t>(dcp::split_cap(T, D, max_seq_len, sms)), 0};
  return dcp::split_workspace_bytes(p, T, H, D) + dcp::order_workspace_bytes(p, T, D);
}

}  // extern "C"

static dcp_status_t decode_partial_impl(const void* q, int64_t q_stride_tok, const void* kv_cache,
                                        dcp_kv_dtype_t kv_dtype, const float* kv_scale,
                                        int32_t num_blocks, int32_t block_size, const int32_t* block_table,
                                        int32_t bt_width, int64_t bt_stride, bool local, int64_t bt_shard_stride,
                                        int32_t d0, int32_t Dn,
                                        const int32_t* seq_lens, const int32_t* query_start_loc, int32_t B,
                                        int32_t T, int32_t H, int32_t max_seq_len, int32_t max_q_len, int32_t D,
                                        int32_t interleave, float scale, void* O_part, dcp_dtype_t o_dtype,
                                        float* lse_part, void* workspace, size_t workspace_bytes, int32_t* dev_error,
                                        void* stream) {
  if (B < 0 || T < 0 || H < 1 || H > 1024 || D < 1 || D > DCP_MAX_SHARDS || interleave < 1 ||
      max_seq_len < 0 || max_q_len < 1 || !std::isfinite(scale))
    return DCP_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return DCP_OK;
  if (!q || !kv_cache || !block_table || !seq_lens || !query_start_loc || !O_part || !lse_part)
    return DCP_ERR_INVALID_ARG;
  if ((kv_dtype != DCP_KV_BF16 && kv_dtype != DCP_KV_FP8_E4M3) || (o_dtype != DCP_DTYPE_F32 && o_dtype != DCP_DTYPE_BF16))
    return DCP_ERR_UNSUPPORTED_DTYPE;
  if (kv_dtype == DCP_KV_FP8_E4M3 && !kv_scale) return DCP_ERR_INVALID_ARG;
  if (num_blocks < 1 || block_size < 1 || bt_width < 1 || bt_stride < bt_width ||
      q_stride_tok < static_cast<int64_t>(H) * DCP_KV_DIM)
    return DCP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(O_part) || (q_stride_tok % 8) != 0)
    return DCP_ERR_MISALIGNED;
  if (d0 < 0 || Dn < 1 || d0 + Dn > D) return DCP_ERR_INVALID_ARG;
  if (local && Dn > 1 && bt_shard_stride < static_cast<int64_t>(B - 1) * bt_stride + bt_width)
    return DCP_ERR_INVALID_ARG;  // shards' tables would overlap
  // a table row covers the longest sequence (global layout) or the largest
  // computed local shard, the first (per-shard layout)
  const int64_t covered = local ? dcp::local_len(max_seq_len, d0, D, interleave) : max_seq_len;
  if ((covered + block_size - 1) / block_size > bt_width) return DCP_ERR_TABLE_TOO_NARROW;

  const DecodeLaunch launch =
      decode_launch(T, H, D, interleave, d0, Dn, max_seq_len, workspace != nullptr, workspace_bytes,
                    kv_dtype == DCP_KV_FP8_E4M3);
  const dcp::SplitPlan plan = launch.plan;
  const size_t need = launch.need;
  if (need > 0 && (workspace_bytes < need || !workspace)) return DCP_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && !aligned16(workspace)) return DCP_ERR_MISALIGNED;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DecodeArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.q_stride_tok = q_stride_tok;
  a.kv = kv_cache;
  a.kv_fp8 = kv_dtype == DCP_KV_FP8_E4M3 ? 1 : 0;
  a.kv_scale = kv_scale;
  a.o_bf16 = o_dtype == DCP_DTYPE_BF16 ? 1 : 0;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.block_table = block_table;
  a.bt_width = bt_width;
  a.bt_stride = bt_stride;
  a.local_tables = local ? 1 : 0;
  a.bt_shard_stride = local ? bt_shard_stride : 0;
  a.seq_lens = seq_lens;
  a.qsl = query_start_loc;
  a.B = B; a.T = T; a.H = H;
  a.max_seq_len = max_seq_len; a.max_q_len = max_q_len;
  // a request's verification rows side by side (when the rows split evenly
  // into groups of max_q_len: a permutation of the units either way)
  a.row_group = (max_q_len >= 2 && max_q_len <= 8 && T % max_q_len == 0) ? max_q_len : 1;
  a.D = D; a.I = interleave;
  a.div_I = dcp::make_fastdiv(interleave);
  a.div_bs = dcp::make_fastdiv(block_size);
  a.d0 = d0; a.Dn = Dn;
  a.scale = scale;
  a.plan = plan;
  a.dev_error = dev_error;
  const char* stall = std::getenv("DCP_TEST_STALL_WAIT");  // failure-path test hook (see DecodeArgs)
  a.stall_test = stall && stall[0] == '1';
  void* ws_O = nullptr;
  float* ws_lse = nullptr;
  if (plan.splits > 1) {
    const size_t pairs = static_cast<size_t>(plan.splits) * Dn * T * H;
    ws_O = workspace;  // split partials in the output's dtype (sized for fp32)
    ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                      (pairs * DCP_LATENT_DIM * sizeof(float) + 255) / 256 * 256);
    a.O_dst = ws_O;
    a.lse_dst = ws_lse;
  } else {
    a.O_dst = O_part;
    a.lse_dst = lse_part;
  }
  const bool simt = launch.simt;
  a.unit_order = nullptr;
  cudaError_t e = cudaSuccess;
  if (launch.use_order) {
    // more units than clusters that fit at once: start the long ones first
    // (the order lives in the workspace past the split partials; a workspace
    // without room for it keeps index order)
    const int64_t units = static_cast<int64_t>(T) * Dn * plan.splits;
    int32_t* order = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + need);
    e = dcp::launch_unit_order(a, static_cast<int32_t>(units), order, st);
    if (e != cudaSuccess) return DCP_ERR_CUDA;
    a.unit_order = order;
  }
  e = simt ? dcp::launch_decode_simt(a, st) : dcp::launch_decode_tc(a, st);
  if (e != cudaSuccess) return DCP_ERR_CUDA;
  if (plan.splits > 1) {
    const int64_t pairs = static_cast<int64_t>(Dn) * T * H;
    e = dcp::launch_lse_merge(ws_O, a.o_bf16 != 0, ws_lse, pairs * DCP_LATENT_DIM, pairs, plan.splits, pairs, H,
                              nullptr, nullptr, 0, /*row_mask=*/false, O_part, a.o_bf16 != 0, lse_part, st);
    if (e != cudaSuccess) return DCP_ERR_CUDA;
  }
  return DCP_OK;
}


extern "C" {

dcp_status_t dcp_mla_decode_partial(const void* q, int64_t q_stride_tok, const void* kv_cache,
                                    int32_t num_blocks, int32_t block_size, const int32_t* block_table,
                                    int32_t bt_width, int64_t bt_stride, const int32_t* seq_lens,
                                    const int32_t* query_start_loc, int32_t B, int32_t T, int32_t H,
                                    int32_t max_seq_len, int32_t max_q_len, int32_t D, int32_t interleave,
                                    float scale, float* O_part, float* lse_part, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_error, void* stream) {
  return decode_partial_impl(q, q_stride_tok, kv_cache, DCP_KV_BF16, nullptr, num_blocks, block_size, block_table,
                             bt_width, bt_stride, false, 0, 0, D, seq_lens, query_start_loc, B, T, H, max_seq_len,
                             max_q_len, D, interleave, scale, O_part, DCP_DTYPE_F32, lse_part, workspace,
                             workspace_bytes, dev_error, stream);
}

dcp_status_t dcp_mla_decode_partial_local(const void* q, int64_t q_stride_tok, const void* kv_cache,
                                          int32_t num_blocks, int32_t block_size, const int32_t* block_table,
                                          int32_t bt_width, int64_t bt_stride, int64_t bt_shard_stride,
                                          const int32_t* seq_lens, const int32_t* query_start_loc, int32_t B,
                                          int32_t T, int32_t H, int32_t max_seq_len, int32_t max_q_len, int32_t D,
                                          int32_t interleave, int32_t shard_begin, int32_t shard_count,
                                          float scale, float* O_part, float* lse_part, void* workspace,
                                          size_t workspace_bytes, int32_t* dev_error, void* stream) {
  return decode_partial_impl(q, q_stride_tok, kv_cache, DCP_KV_BF16, nullptr, num_blocks, block_size, block_table,
                             bt_width, bt_stride, true, bt_shard_stride, shard_begin, shard_count, seq_lens,
                             query_start_loc, B, T, H, max_seq_len, max_q_len, D, interleave, scale, O_part,
                             DCP_DTYPE_F32, lse_part, workspace, workspace_bytes, dev_error, stream);
}

dcp_status_t dcp_mla_decode_partial_v2(const void* q, int64_t q_stride_tok, const void* kv_cache,
                                       dcp_kv_dtype_t kv_dtype, const float* kv_scale, int32_t num_blocks,
                                       int32_t block_size, const int32_t* block_table, int32_t bt_width,
                                       int64_t bt_stride, int32_t per_shard_tables, int64_t bt_shard_stride,
                                       int32_t shard_begin, int32_t shard_count, const int32_t* seq_lens,
                                       const int32_t* query_start_loc, int32_t B, int32_t T, int32_t H,
                                       int32_t max_seq_len, int32_t max_q_len, int32_t D, int32_t interleave,
                                       float scale, void* O_part, dcp_dtype_t o_dtype, float* lse_part,
                                       void* workspace, size_t workspace_bytes, int32_t* dev_error, void* stream) {
  return decode_partial_impl(q, q_stride_tok, kv_cache, kv_dtype, kv_scale, num_blocks, block_size, block_table,
                             bt_width, bt_stride, per_shard_tables != 0, bt_shard_stride, shard_begin, shard_count,
                             seq_lens, query_start_loc, B, T, H, max_seq_len, max_q_len, D, interleave, scale, O_part,
                             o_dtype, lse_part, workspace, workspace_bytes, dev_error, stream);
}

int32_t dcp_decode_kernel_launches(int32_t B, int32_t T, int32_t H, int32_t D, int32_t interleave,
                                   int32_t max_seq_len, int32_t max_q_len, size_t workspace_bytes) {
  if (B < 0 || T < 0 || H < 1 || H > 1024 || D < 1 || D > DCP_MAX_SHARDS || interleave < 1 || max_seq_len < 0 ||
      max_q_len < 0)
    return -1;
  if (B == 0 || T == 0) return 0;
  const DecodeLaunch L =
      decode_launch(T, H, D, interleave, 0, D, max_seq_len, workspace_bytes > 0, workspace_bytes);
  return 1 + (L.plan.splits > 1 ? 1 : 0) + (L.use_order ? 1 : 0);
}

static dcp_status_t combine_impl(const void* O_part, dcp_dtype_t part_dtype, const float* lse_part,
                                 const int32_t* seq_lens, const int32_t* query_start_loc, int32_t B, int32_t T,
                                 int32_t H, int32_t D, void* out, dcp_dtype_t out_dtype, float* out_lse,
                                 void* stream) {
  if (B < 0 || T < 0 || H < 1 || D < 1 || D > DCP_MAX_SHARDS) return DCP_ERR_INVALID_ARG;
  if ((out_dtype != DCP_DTYPE_BF16 && out_dtype != DCP_DTYPE_F32) ||
      (part_dtype != DCP_DTYPE_BF16 && part_dtype != DCP_DTYPE_F32))
    return DCP_ERR_UNSUPPORTED_DTYPE;
  if (B == 0 || T == 0) return DCP_OK;
  if (!O_part || !lse_part || !seq_lens || !query_start_loc || !out || !out_lse)
    return DCP_ERR_INVALID_ARG;
  if (!aligned16(O_part) || !aligned16(out)) return DCP_ERR_MISALIGNED;
  const int64_t pairs = static_cast<int64_t>(T) * H;
  // out must not overlap O_part
  const char* ob = static_cast<const char*>(out);
  const char* oe = ob + pairs * DCP_LATENT_DIM * (out_dtype == DCP_DTYPE_BF16 ? 2 : 4);
  const char* pb = static_cast<const char*>(O_part);
  const char* pe = pb + static_cast<int64_t>(D) * pairs * DCP_LATENT_DIM * (part_dtype == DCP_DTYPE_BF16 ? 2 : 4);
  if (ob < pe && pb < oe) return DCP_ERR_INVALID_ARG;
  const cudaError_t e = dcp::launch_lse_merge(O_part, part_dtype == DCP_DTYPE_BF16, lse_part, pairs * DCP_LATENT_DIM,
                                              pairs, D, pairs, H, seq_lens, query_start_loc, B, /*row_mask=*/true,
                                              out, out_dtype == DCP_DTYPE_BF16, out_lse, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}

dcp_status_t dcp_lse_combine(const float* O_part, const float* lse_part, const int32_t* seq_lens,
                             const int32_t* query_start_loc, int32_t B, int32_t T, int32_t H, int32_t D,
                             void* out, dcp_dtype_t out_dtype, float* out_lse, void* stream) {
  return combine_impl(O_part, DCP_DTYPE_F32, lse_part, seq_lens, query_start_loc, B, T, H, D, out, out_dtype, out_lse,
                      stream);
}

dcp_status_t dcp_lse_combine_v2(const void* O_part, dcp_dtype_t part_dtype, const float* lse_part,
                                const int32_t* seq_lens, const int32_t* query_start_loc, int32_t B, int32_t T,
                                int32_t H, int32_t D, void* out, dcp_dtype_t out_dtype, float* out_lse,
                                void* stream) {
  return combine_impl(O_part, part_dtype, lse_part, seq_lens, query_start_loc, B, T, H, D, out, out_dtype, out_lse,
                      stream);
}

dcp_status_t dcp_decode_concat_cache(const void* ql_nope, int64_t ql_nope_stride_tok, int64_t ql_nope_stride_head,
                                     const void* q_pe, int64_t q_pe_stride_tok, int64_t q_pe_stride_head,
                                     const void* kv_c, int64_t kv_c_stride_tok, const void* k_pe,
                                     int64_t k_pe_stride_tok, const int64_t* slot_mapping, int32_t T, int32_t H,
                                     void* q_out, int64_t q_out_stride_tok, void* kv_cache, int64_t num_slots,
                                     int32_t* dev_error, void* stream) {
  if (T < 0 || H < 1 || num_slots < 1) return DCP_ERR_INVALID_ARG;
  if (T == 0) return DCP_OK;
  if (!ql_nope || !q_pe || !kv_c || !k_pe || !slot_mapping || !q_out || !kv_cache) return DCP_ERR_INVALID_ARG;
  if (ql_nope_stride_tok < 0 || ql_nope_stride_head < 0 || q_pe_stride_tok < 0 || q_pe_stride_head < 0 ||
      kv_c_stride_tok < 0 || k_pe_stride_tok < 0 || q_out_stride_tok < static_cast<int64_t>(H) * DCP_KV_DIM)
    return DCP_ERR_INVALID_ARG;
  const int64_t strides[] = {ql_nope_stride_tok, ql_nope_stride_head, q_pe_stride_tok, q_pe_stride_head,
                             kv_c_stride_tok,    k_pe_stride_tok,     q_out_stride_tok};
  for (int64_t st : strides)
    if (st % 8 != 0) return DCP_ERR_MISALIGNED;  // 16-byte units
  if (!aligned16(ql_nope) || !aligned16(q_pe) || !aligned16(kv_c) || !aligned16(k_pe) || !aligned16(q_out) ||
      !aligned16(kv_cache))
    return DCP_ERR_MISALIGNED;
  dcp::ConcatCacheArgs a{};
  a.ql_nope = ql_nope; a.ql_nope_stride_tok = ql_nope_stride_tok; a.ql_nope_stride_head = ql_nope_stride_head;
  a.q_pe = q_pe; a.q_pe_stride_tok = q_pe_stride_tok; a.q_pe_stride_head = q_pe_stride_head;
  a.kv_c = kv_c; a.kv_c_stride_tok = kv_c_stride_tok;
  a.k_pe = k_pe; a.k_pe_stride_tok = k_pe_stride_tok;
  a.slot_mapping = slot_mapping;
  a.T = T; a.H = H;
  a.q_out = q_out; a.q_out_stride_tok = q_out_stride_tok;
  a.kv_cache = kv_cache; a.num_slots = num_slots;
  a.dev_error = dev_error;
  return dcp::launch_concat_cache(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}

}  // extern "C"
