// Shared device/host helpers of the DCP MLA hot path: row resolution, the
// token -> shard mapper and the paged block-table walker.  Integer only; the
// same inline functions back the host-visible dcp_shard_of/dcp_local_len.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/dcp.h"

#define DCP_HD __host__ __device__ __forceinline__

namespace dcp {

constexpr int kLatent = DCP_LATENT_DIM;  // 512 value dims
constexpr int kRope = DCP_ROPE_DIM;      // 64 rope dims
constexpr int kKDim = DCP_KV_DIM;        // 576 = one latent row / one query head row
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Tokens are dealt to D shards round-robin in runs of I
// (cp_kv_cache_interleave_size) ["[Kimi-K3] DCP support" summary on
// prhub.com.cn, implementation step 3].
DCP_HD int32_t shard_of(int64_t pos, int32_t D, int32_t I) {
  return static_cast<int32_t>((pos / I) % D);
}

// |{p < L : shard_of(p) == d}| in closed form.
DCP_HD int32_t local_len(int32_t L, int32_t d, int32_t D, int32_t I) {
  const int64_t period = static_cast<int64_t>(I) * D;
  const int64_t full = L / period;
  int64_t rem = L % period - static_cast<int64_t>(d) * I;
  rem = rem < 0 ? 0 : (rem > I ? I : rem);
  return static_cast<int32_t>(full * I + rem);
}

// Global position of shard d's j-th token (inverse of the mapper).
DCP_HD int64_t local_to_global(int64_t j, int32_t d, int32_t D, int32_t I) {
  return (j / I) * (static_cast<int64_t>(D) * I) + static_cast<int64_t>(d) * I + j % I;
}

// Request owning query row r: the b with qsl[b] <= r < qsl[b+1], or -1 when
// r lies before qsl[0] or at/after qsl[B].  qsl is non-decreasing.
__device__ __forceinline__ int32_t find_request(const int32_t* __restrict__ qsl, int32_t B, int32_t r) {
  if (B <= 0 || r < __ldg(qsl) || r >= __ldg(qsl + B)) return -1;
  int32_t lo = 0, hi = B;  // invariant: qsl[lo] <= r < qsl[hi]
  while (hi - lo > 1) {
    const int32_t mid = (lo + hi) >> 1;
    if (__ldg(qsl + mid) <= r) lo = mid; else hi = mid;
  }
  return lo;
}

struct RowInfo {
  int32_t b;        // request, -1 if none
  int32_t L;        // the row's own context length (0 for padding rows)
  bool padding;     // no request, or a seq_len == 0 request
  uint32_t err;     // DCP_DEVERR_* bits seen while resolving
};

// Row resolution: row i of a q_len-row request sees seq_len - (q_len-1-i)
// tokens, formed before any per-shard localisation ("[Kimi-K3] DCP support",
// merged GLM-5.2 DCP+MTP bugfix text: per-token seq_lens are localised after
// the MTP expansion).  seq_len is clamped to max_seq_len (flagged).
__device__ __forceinline__ RowInfo resolve_row(const int32_t* __restrict__ seq_lens,
                                               const int32_t* __restrict__ qsl, int32_t B,
                                               int32_t r, int32_t max_seq_len, int32_t max_q_len) {
  RowInfo ri{-1, 0, true, 0u};
  const int32_t b = find_request(qsl, B, r);
  if (b < 0) return ri;
  ri.b = b;
  int32_t seq = __ldg(seq_lens + b);
  if (seq <= 0) return ri;  // CUDA-graph padding request (negative: treated alike)
  const int32_t q0 = __ldg(qsl + b), q1 = __ldg(qsl + b + 1);
  const int32_t q_len = q1 - q0;
  if (q_len > max_q_len) ri.err |= DCP_DEVERR_BAD_ROWS;
  if (seq > max_seq_len) { ri.err |= DCP_DEVERR_SEQ_TOO_LONG; seq = max_seq_len; }
  const int32_t L = seq - (q_len - 1 - (r - q0));
  ri.L = L > 0 ? L : 0;
  ri.padding = false;
  return ri;
}

// Combine-side padding test: a row is padding when it has no request or its
// request has seq_len == 0 ("[Kimi-K3] DCP support", CUDA-graph padding
// follow-up and the review thread on the seq_lens == 0 row mask).
__device__ __forceinline__ bool row_is_padding(const int32_t* __restrict__ seq_lens,
                                               const int32_t* __restrict__ qsl, int32_t B, int32_t r) {
  const int32_t b = find_request(qsl, B, r);
  return b < 0 || __ldg(seq_lens + b) <= 0;
}

// Split-KV plan shared by the workspace query and the launch: each (row,
// shard) pair's local tokens are cut into `splits` ranges of `chunk` tokens.
struct SplitPlan {
  int32_t splits;
  int32_t chunk;
};

SplitPlan plan_splits(int32_t T, int32_t D, int32_t I, int32_t max_seq_len, int sm_count);

}  // namespace dcp
