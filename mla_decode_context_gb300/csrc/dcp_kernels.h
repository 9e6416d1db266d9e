// Internal launch interface between the C ABI (dcp_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "dcp_common.cuh"

namespace dcp {

// Division of a non-negative int32 n < 2^31 by a positive int32 d fixed for
// a launch, as a multiply-high, an add and a shift (the round-up method of
// Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1 (which fits in 32 bits),
// n / d = (umulhi(n, m) + n) >> l, the sum staying below 2^32.
struct FastDiv {
  uint32_t d, m, l;
};
inline FastDiv make_fastdiv(int32_t d) {
  FastDiv f{static_cast<uint32_t>(d), 0u, 0u};
  while ((1ull << f.l) < f.d) ++f.l;
  f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.l) - f.d)) / f.d + 1);
  return f;
}
#ifdef __CUDACC__
__device__ __forceinline__ int32_t fast_div(int32_t n, const FastDiv& f) {
  const uint32_t u = static_cast<uint32_t>(n);
  return static_cast<int32_t>((__umulhi(u, f.m) + u) >> f.l);
}
#endif

// Everything one decode launch needs (validated by the C ABI).
struct DecodeArgs {
  const __nv_bfloat16* q;
  int64_t q_stride_tok;  // elements between consecutive rows of q
  // latent cache rows: bf16 [576], or (kv_fp8) FP8 E4M3 codes [576] whose
  // values are code x kv_scale[row] (one fp32 scale per cache slot)
  const void* kv;
  int32_t kv_fp8;
  const float* kv_scale;
  int32_t num_blocks, block_size;
  const int32_t* block_table;
  int32_t bt_width;
  int64_t bt_stride;        // elements between requests' table rows
  // per-shard (rank-local) tables: block_table is [D, B, W] with shard d's
  // rows bt_shard_stride elements after shard d - 1's, and shard d's j-th
  // local token lives in row table[d, b, j / block_size] * block_size +
  // j % block_size; otherwise one table row per request over positions
  int32_t local_tables;
  int64_t bt_shard_stride;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int32_t B, T, H, max_seq_len, max_q_len, D, I;
  FastDiv div_I, div_bs;  // division by I and by block_size (set with them)
  // the shards this launch computes: d0 .. d0 + Dn - 1 (all D on one GPU;
  // one per rank when each DCP rank holds only its own shard).  Outputs and
  // per-shard tables are indexed by d - d0.
  int32_t d0, Dn;
  float scale;
  // Where partials go: O_dst[((s * Dn + d - d0) * T + r) * H + h][512] with s
  // the split (s == 0 only when splits == 1, then O_dst = O_part).
  void* O_dst;      // fp32, or bf16 when o_bf16
  int32_t o_bf16;
  float* lse_dst;
  SplitPlan plan;
  int32_t* dev_error;
  // Optional launch order of the tensor-core decode's units (cluster c runs
  // unit unit_order[c]); nullptr = index order.
  const int32_t* unit_order;
  // Rows per group of the unit index (1, or the verification width when
  // every request has that many rows): see unit_coords.
  int32_t row_group;
  // Test hook for the failure path (0 in normal use): nonzero makes the
  // tensor-core decode's first softmax group wait on a barrier that nothing
  // completes, so every unit ends through its bounded waits and reports
  // DCP_DEVERR_TIMEOUT.
  int32_t stall_test;
};

// The (row, shard - d0, split) of unit u of the tensor-core decode, with the
// rows of each group of row_group consecutive rows innermost: u = ((row /
// row_group x Dn + shard - d0) x splits + split) x row_group + row %
// row_group.  With row_group = the requests' verification width, a request's
// rows for one (shard, split) run side by side and read each KV tile from L2
// at the same time, so the request's KV comes from HBM about once.
struct UnitCoords {
  int32_t r, dd, s;
};
__device__ __forceinline__ UnitCoords unit_coords(const DecodeArgs& a, int64_t u) {
  const int64_t g = a.row_group > 1 ? a.row_group : 1;
  const int64_t i = u % g, rest = u / g;
  const int32_t s = static_cast<int32_t>(rest % a.plan.splits);
  const int64_t rest2 = rest / a.plan.splits;
  const int32_t dd = static_cast<int32_t>(rest2 % a.Dn);
  return UnitCoords{static_cast<int32_t>((rest2 / a.Dn) * g + i), dd, s};
}

// Generic LSE merge over `nsrc` sources: pair p (flattened) reads
// lse_src[s * lse_stride + p] and O_src[s * o_stride + p * 512 ...] (fp32, or
// bf16 with src_bf16), and writes out[p * 512 ...] (fp32, or bf16 with
// out_bf16, round to nearest even) and out_lse[p].  With row masking, pair p
// belongs to row p / H and padding rows give 0 / -inf.
cudaError_t launch_lse_merge(const void* O_src, bool src_bf16, const float* lse_src, int64_t o_stride,
                             int64_t lse_stride, int nsrc, int64_t npairs, int32_t H, const int32_t* seq_lens,
                             const int32_t* qsl, int32_t B, bool row_mask, void* out, bool out_bf16,
                             float* out_lse, cudaStream_t st);

// Reference SIMT decode (fp32 FMA, any geometry).
cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t st);

// The decode step before attention: query concat and paged-cache write
// (validated by the C ABI; strides in elements, 16-byte aligned).
struct ConcatCacheArgs {
  const void* ql_nope;  // bf16 [T, H, 512]
  int64_t ql_nope_stride_tok, ql_nope_stride_head;
  const void* q_pe;     // bf16 [T, H, 64]
  int64_t q_pe_stride_tok, q_pe_stride_head;
  const void* kv_c;     // bf16 [T, 512]
  int64_t kv_c_stride_tok;
  const void* k_pe;     // bf16 [T, 64]
  int64_t k_pe_stride_tok;
  const int64_t* slot_mapping;  // [T]
  int32_t T, H;
  void* q_out;          // bf16 [T, H, 576]
  int64_t q_out_stride_tok;
  void* kv_cache;       // bf16 [num_slots, 576]
  int64_t num_slots;
  int32_t* dev_error;
};
cudaError_t launch_concat_cache(const ConcatCacheArgs& a, cudaStream_t st);

// Tensor-core decode (tcgen05/TMEM/TMA, 2-CTA clusters).  Supported when
// H <= 128 and the shard layout tiles into whole TMA boxes: block_size a
// multiple of D * interleave (runs inside blocks) or interleave a multiple
// of block_size (whole blocks per run).
// Writes into `order` the units (row, shard, split) of `a` sorted by
// decreasing 1 + floor(log2(tiles)), stable in unit index, so that long units
// start first when there are more units than clusters that fit at once.
cudaError_t launch_unit_order(const DecodeArgs& a, int32_t units, int32_t* order, cudaStream_t st);

bool decode_tc_supported(const DecodeArgs& a);
// CTAs of the tensor-core decode resident at once on the current device
// (0 if unknown); the split plan sizes one wave from it.
int decode_tc_resident_ctas();
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st);

}  // namespace dcp
