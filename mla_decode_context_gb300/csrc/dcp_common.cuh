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

// The request owning query row r, with its row range and seq_len: b is the
// request with qsl[b] <= r < qsl[b+1] (unique: qsl is non-decreasing), or -1
// when r lies before qsl[0] or at/after qsl[B].  Batches whose requests all
// have the same number of rows (one decode row each, or a fixed verification
// width) resolve in two rounds of independent loads: the guess
// g = (r - qsl[0]) / (qsl[1] - qsl[0]) is checked against qsl[g], qsl[g+1]
// (loaded together with seq_lens[g]); any other layout falls back to a
// binary search.
struct RequestOfRow {
  int32_t b;       // -1 if none
  int32_t q0, q1;  // qsl[b], qsl[b+1]
  int32_t seq;     // seq_lens[b]
};

// width_hint > 0: a guess of the rows per request (requests of equal width
// from row 0), whose entries are read together with the bounds, so that the
// common case costs one round of loads instead of two; the guess is used
// only when qsl confirms it.
__device__ __forceinline__ RequestOfRow request_of_row(const int32_t* __restrict__ seq_lens,
                                                       const int32_t* __restrict__ qsl, int32_t B, int32_t r,
                                                       int32_t width_hint = 0) {
  RequestOfRow q{-1, 0, 0, 0};
  if (B <= 0) return q;
  const int32_t gh = width_hint > 0 ? min(max(r, 0) / width_hint, B - 1) : 0;
  const int32_t qa = __ldg(qsl), qn = __ldg(qsl + 1), qB = __ldg(qsl + B);
  int32_t hlo = 0, hhi = 0, hsq = 0;
  if (width_hint > 0) hlo = __ldg(qsl + gh), hhi = __ldg(qsl + gh + 1), hsq = __ldg(seq_lens + gh);
  if (r < qa || r >= qB) return q;
  if (width_hint > 0 && hlo <= r && r < hhi) return RequestOfRow{gh, hlo, hhi, hsq};
  const int32_t step = qn - qa;
  if (step > 0) {
    const int32_t g = (r - qa) / step;
    if (g < B) {
      const int32_t lo = __ldg(qsl + g), hi = __ldg(qsl + g + 1), sq = __ldg(seq_lens + g);
      if (lo <= r && r < hi) return RequestOfRow{g, lo, hi, sq};
    }
  }
  int32_t lo = 0, hi = B;  // invariant: qsl[lo] <= r < qsl[hi]
  while (hi - lo > 1) {
    const int32_t mid = (lo + hi) >> 1;
    if (__ldg(qsl + mid) <= r) lo = mid; else hi = mid;
  }
  return RequestOfRow{lo, __ldg(qsl + lo), __ldg(qsl + lo + 1), __ldg(seq_lens + lo)};
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
  const RequestOfRow q = request_of_row(seq_lens, qsl, B, r, max_q_len);
  if (q.b < 0) return ri;
  ri.b = q.b;
  int32_t seq = q.seq;
  if (seq <= 0) return ri;  // CUDA-graph padding request (negative: treated alike)
  const int32_t q_len = q.q1 - q.q0;
  if (q_len > max_q_len) ri.err |= DCP_DEVERR_BAD_ROWS;
  if (seq > max_seq_len) { ri.err |= DCP_DEVERR_SEQ_TOO_LONG; seq = max_seq_len; }
  const int32_t L = seq - (q_len - 1 - (r - q.q0));
  ri.L = L > 0 ? L : 0;
  ri.padding = false;
  return ri;
}

// Combine-side padding test: a row is padding when it has no request or its
// request has seq_len == 0 ("[Kimi-K3] DCP support", CUDA-graph padding
// follow-up and the review thread on the seq_lens == 0 row mask).
__device__ __forceinline__ bool row_is_padding(const int32_t* __restrict__ seq_lens,
                                               const int32_t* __restrict__ qsl, int32_t B, int32_t r) {
  const RequestOfRow q = request_of_row(seq_lens, qsl, B, r);
  return q.b < 0 || q.seq <= 0;
}

// Split-KV plan shared by the workspace query and the launch: each (row,
// shard) pair's local tokens are cut into `splits` ranges of `chunk` tokens.
struct SplitPlan {
  int32_t splits;
  int32_t chunk;
};

// D, I: the interleave rule; [d0, d0 + Dn): the shards computed.
SplitPlan plan_splits(int32_t T, int32_t D, int32_t I, int32_t d0, int32_t Dn, int32_t max_seq_len, int sm_count);

}  // namespace dcp
