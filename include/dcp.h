/*
 * dcp.h - C ABI of the GB300 (sm_103a) decode-context-parallel MLA hot path.
 *
 * Decode context parallelism (DCP) splits each request's KV context over D
 * shards; every shard runs absorbed-MLA decode attention over its own tokens
 * and returns a partial output plus its log-sum-exp, and an LSE-weighted
 * combine merges the shards.  On one GPU the D shards are D disjoint token
 * partitions of one paged latent KV cache resident in HBM.
 *
 * Sources (pages on the method):
 *   [PR50484] "[Kimi-K3] DCP support", vllm-project/vllm pull request 50484:
 *             Summary (empty-KV-shard masking of the LSE-weighted reduction),
 *             "CUDA-graph padding follow-up" and the review thread on the
 *             padding-row mask (rows of seq_len == 0 requests).
 *   [PRHUB]   prhub.com.cn summary of the same pull request: implementation
 *             steps 3-4 (interleaved DCP chunking; -inf masking at the source;
 *             exp2 LSE-weighted merge; zero-weight skip at the consumer;
 *             16-byte row alignment), key snippet "Decode: latent multi-query
 *             attention" (forward_mqa returns (latent_out, lse); then
 *             combine(latent_out, lse, seq_lens, query_start_loc)), risk 2
 *             (unsupported dtypes are rejected) and risk 4 (timeouts trap in
 *             the pages' kernel; here they return a status).
 *   [PR565]   "perf(mla): fuse K3 DCP verification queries",
 *             local-inference-lab/vllm pull request 565: Summary (the K=3
 *             verification rows share each KV load) and review follow-up
 *             (block-table width contract; reject a table narrower than the
 *             largest local shard).
 *
 * Conventions shared by every entry point:
 *   - All pointers to arrays are DEVICE pointers to caller-owned memory on the
 *     current CUDA device; the library allocates nothing, keeps no state
 *     between calls, never synchronises, and enqueues its kernels on
 *     `stream` (a cudaStream_t; NULL = legacy default stream).  A call
 *     returns DCP_OK once its kernels are enqueued.
 *   - Arrays are dense row-major unless a stride argument says otherwise.
 *     Strides are in ELEMENTS.
 *   - Host-detectable errors return a status before anything is launched.
 *     Errors only the device can see (a block id outside the cache, a
 *     sequence longer than the declared maximum) never trap: the kernel skips
 *     the offending token and ORs a DCP_DEVERR_* bit into *dev_error when
 *     dev_error is non-NULL.
 *   - Latent geometry is fixed: a KV cache row and a query head row are
 *     DCP_KV_DIM = 576 bf16 values (512 compressed-KV dims followed by 64
 *     rope dims); values are the first DCP_LATENT_DIM = 512 dims.
 *   - LSEs are natural logarithms; -inf marks "no tokens".
 *   - Two environment variables, read on every call and unset in normal use,
 *     change what dcp_mla_decode_partial runs:
 *       DCP_FORCE_SIMT=1       the CUDA-core reference kernel instead of the
 *                              tensor-core one (A/B checks);
 *       DCP_TEST_STALL_WAIT=1  test hook for the failure path: one wait of
 *                              the tensor-core kernel runs out on purpose
 *                              (on a barrier nothing completes), so the call
 *                              ends with DCP_DEVERR_TIMEOUT in *dev_error
 *                              after about a second per bounded wait; the
 *                              outputs are undefined.
 */
#ifndef DCP_H_
#define DCP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DCP_LATENT_DIM 512
#define DCP_ROPE_DIM 64
#define DCP_KV_DIM 576
#define DCP_MAX_SHARDS 32

/* Device-side error bits ORed into *dev_error. */
#define DCP_DEVERR_BAD_BLOCK 1    /* a referenced block id is outside [0, num_blocks) */
#define DCP_DEVERR_SEQ_TOO_LONG 2 /* seq_len > max_seq_len (clamped to max_seq_len) */
#define DCP_DEVERR_BAD_ROWS 4     /* query_start_loc decreasing, or q_len > max_q_len */
#define DCP_DEVERR_TIMEOUT 8      /* a bounded on-device wait gave up */

typedef enum {
  DCP_OK = 0,
  DCP_ERR_INVALID_ARG = 1,       /* null pointer, negative or inconsistent size */
  DCP_ERR_UNSUPPORTED_DTYPE = 2, /* output dtype not supported [PRHUB, risk 2] */
  DCP_ERR_MISALIGNED = 3,        /* pointer or row stride not 16-byte aligned [PRHUB, step 4] */
  DCP_ERR_TABLE_TOO_NARROW = 4,  /* bt_width < ceil(max_seq_len / block_size) [PR565, review follow-up] */
  DCP_ERR_WORKSPACE_TOO_SMALL = 5,
  DCP_ERR_CUDA = 6,              /* a CUDA runtime/driver call failed (launch, attribute query) */
  DCP_ERR_TIMEOUT = 7            /* reserved for bounded cross-device waits */
} dcp_status_t;

typedef enum { DCP_DTYPE_BF16 = 0, DCP_DTYPE_F32 = 1 } dcp_dtype_t;

/* Latent KV cache formats: bf16 rows, or FP8 E4M3 codes (1 sign, 4 exponent
 * bits with bias 7, 3 mantissa bits; no infinity) with one fp32 scale per
 * cache slot (value = code x scale) ["perf(mla): fuse K3 DCP verification
 * queries", review follow-up: fp8 KV verify plans]. */
typedef enum { DCP_KV_BF16 = 0, DCP_KV_FP8_E4M3 = 1 } dcp_kv_dtype_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* dcp_status_str(dcp_status_t status);

/* Library ABI version (increments when a signature changes). */
int dcp_version(void);

/*
 * Token -> shard mapper (host copy of the device code, for tests).
 * Positions are dealt to the D shards round-robin in runs of `interleave`
 * tokens (cp_kv_cache_interleave_size): shard(pos) = floor(pos / I) mod D
 * [PRHUB, implementation step 3].  Returns -1 if D < 1, I < 1 or pos < 0.
 */
int32_t dcp_shard_of(int64_t pos, int32_t D, int32_t interleave);

/*
 * How many of the first L positions shard d owns:
 *   floor(L / (I D)) * I + clamp(L mod (I D) - d I, 0, I).
 * Returns -1 on invalid arguments (L < 0, d outside [0, D), D < 1, I < 1).
 */
int32_t dcp_local_len(int32_t L, int32_t d, int32_t D, int32_t interleave);

/*
 * Bytes of device workspace dcp_mla_decode_partial should get for these sizes
 * on the CURRENT device (the split-KV plan depends on its SM count): the
 * split partials plus one int32 per work unit for the order in which the
 * units start (long ones first when they do not all fit on the GPU at once).
 * A workspace that covers only the split partials is accepted (units then
 * start in index order); with no split partials it may be NULL.  Returns
 * (size_t)-1 on invalid arguments.
 */
size_t dcp_decode_workspace_size(int32_t B, int32_t T, int32_t H, int32_t D,
                                 int32_t max_seq_len, int32_t max_q_len);

/*
 * Number of kernels one dcp_mla_decode_partial call with these sizes and this
 * workspace size launches on the CURRENT device: the decode, plus the merge of
 * the split partials when the long-context split is used, plus the ordering
 * of the work units when there are more of them than fit on the GPU at once
 * (and the workspace has room for it).  0 when B or T is 0; -1 on invalid
 * arguments.  For callers that count or capture launches; no page has a
 * counterpart.
 */
int32_t dcp_decode_kernel_launches(int32_t B, int32_t T, int32_t H, int32_t D, int32_t interleave,
                                   int32_t max_seq_len, int32_t max_q_len, size_t workspace_bytes);

/*
 * Absorbed-MLA decode attention split over D context shards.
 * [PRHUB, snippet "Decode: latent multi-query attention": forward_mqa(q,
 *  kv_cache, metadata) -> (latent_out, lse) per rank's shard;
 *  PR50484 Summary and PRHUB step 4: empty shards masked to -inf at source;
 *  PR565 Summary: verification rows of one request share each KV load.]
 *
 * For query row r of request b (rows qsl[b] .. qsl[b+1]-1, q_len = their
 * count, i = r - qsl[b]) the row's own context length is
 *   L_r = max(0, seq_lens[b] - (q_len - 1 - i))
 * (the new tokens are already in the cache).  For each shard d and head h:
 *   S = { p < L_r : floor(p / interleave) mod D == d }
 *   s_p = scale * sum_{k<576} q[r,h,k] * kv(p)[k]
 *   lse_part[d,r,h] = ln sum_{p in S} exp(s_p)
 *   O_part[d,r,h,v] = sum_{p in S} exp(s_p - lse_part[d,r,h]) * kv(p)[v],  v < 512
 * where kv(p) is cache row block_table[b, p / block_size] * block_size +
 * p % block_size.  If S is empty, the row is a padding row (seq_lens[b] == 0)
 * or r >= qsl[B]: lse_part = -inf and O_part = 0, and no KV is read.
 *
 *   q               bf16 [T, H, 576]; row r starts at q + r * q_stride_tok
 *                   (q_stride_tok >= H * 576, a multiple of 8).
 *   kv_cache        bf16 [num_blocks, block_size, 576], dense.
 *   block_table     int32 [B, bt_width], row stride bt_stride (>= bt_width);
 *                   only columns < ceil(L_r / block_size) are read.
 *   seq_lens        int32 [B]; 0 marks a CUDA-graph padding request.
 *   query_start_loc int32 [B + 1], non-decreasing, qsl[0] = 0.
 *   B, T            requests and query rows (rows past qsl[B] are padding).
 *   H               heads (1 .. 1024).
 *   max_seq_len     host-known upper bound of seq_lens (sizes the split plan
 *                   and the table-width check).
 *   max_q_len       host-known upper bound of rows per request.
 *   D, interleave   shard count (1 .. 32) and run length (>= 1).
 *   scale           softmax scale (1/sqrt(192) for Kimi-K3).
 *   O_part          fp32 [D, T, H, 512] output.
 *   lse_part        fp32 [D, T, H] output.
 *   workspace       device scratch of >= dcp_decode_workspace_size(...) bytes,
 *                   16-byte aligned; its contents on entry are ignored.
 *   dev_error       optional int32 device word for DCP_DEVERR_* bits.
 *   stream          cudaStream_t.
 *
 * B == 0 or T == 0 returns DCP_OK without launching anything.
 */
dcp_status_t dcp_mla_decode_partial(
    const void* q, int64_t q_stride_tok,
    const void* kv_cache, int32_t num_blocks, int32_t block_size,
    const int32_t* block_table, int32_t bt_width, int64_t bt_stride,
    const int32_t* seq_lens, const int32_t* query_start_loc,
    int32_t B, int32_t T, int32_t H, int32_t max_seq_len, int32_t max_q_len,
    int32_t D, int32_t interleave, float scale,
    float* O_part, float* lse_part,
    void* workspace, size_t workspace_bytes,
    int32_t* dev_error, void* stream);

/*
 * LSE-weighted combine of D shard partials, with empty-shard and padding-row
 * masking [PRHUB step 4 "exp2 LSE weighted merge"; PR50484 "CUDA-graph
 * padding follow-up"].
 *
 * For each row r and head h: a row whose request has seq_lens == 0 (or that
 * lies past qsl[B]) is a padding row: out = 0, out_lse = -inf, nothing else
 * read.  Otherwise E = { d : lse_part[d,r,h] != -inf }; if E is empty the
 * result is 0 / -inf.  Else, with l_d = lse_part[d,r,h] * log2(e) and
 * M = max_{d in E} l_d:
 *   w_d = exp2(l_d - M),  out = sum_E w_d O_part[d,r,h,:] / sum_E w_d,
 *   out_lse = (M + log2 sum_E w_d) / log2(e).
 * O_part[d,r,h,:] is not read for d outside E (it may hold stale data/NaN).
 *
 *   O_part     fp32 [D, T, H, 512], 16-byte aligned.
 *   lse_part   fp32 [D, T, H].
 *   seq_lens, query_start_loc, B, T: as for the decode call.
 *   H, D       heads (>= 1), shards (1 .. 32).
 *   out        [T, H, 512] of out_dtype (BF16: round to nearest even; F32),
 *              16-byte aligned; must not overlap O_part.
 *   out_lse    fp32 [T, H]; may alias lse_part (the shard-0 slice): every
 *              LSE of a (row, head) is read before its out_lse is written.
 *
 * B == 0 or T == 0 returns DCP_OK without launching anything.
 */
dcp_status_t dcp_lse_combine(
    const float* O_part, const float* lse_part,
    const int32_t* seq_lens, const int32_t* query_start_loc,
    int32_t B, int32_t T, int32_t H, int32_t D,
    void* out, dcp_dtype_t out_dtype, float* out_lse, void* stream);

/*
 * dcp_mla_decode_partial over per-shard (DCP rank-local) block tables: each
 * shard stores only the tokens it owns, densely and in order, in its own
 * blocks, as each rank's own cache does ["[Kimi-K3] DCP support", Summary:
 * each DCP rank keeps its slice of the context; PR565, review follow-up: the
 * plan's page table must cover the largest local KV shard].  Same
 * arguments, results and errors as dcp_mla_decode_partial, except:
 *
 *   shard_begin, shard_count
 *                   the shards this call computes, [shard_begin, shard_begin +
 *                   shard_count) of D (0 <= shard_begin, 1 <= shard_count,
 *                   shard_begin + shard_count <= D, else DCP_ERR_INVALID_ARG):
 *                   all D when one GPU holds every shard, one per DCP rank
 *                   when each rank holds only its own.  D and interleave
 *                   still define which tokens each shard owns.
 *   O_part, lse_part
 *                   fp32 [shard_count, T, H, 512] and [shard_count, T, H].
 *   block_table     int32 [shard_count, B, bt_width]: shard d's j-th local
 *                   token of request b lives in cache row
 *                   table[d - shard_begin, b, j / block_size] * block_size +
 *                   j % block_size.
 *                   Request rows are bt_stride elements apart (>= bt_width),
 *                   shard tables bt_shard_stride apart (with more than one
 *                   shard >= (B - 1) * bt_stride + bt_width, else
 *                   DCP_ERR_INVALID_ARG).  Only the columns a shard's local
 *                   tokens reach are read.
 *   bt_width        must cover the largest computed local shard, the first:
 *                   ceil(local_len(max_seq_len, shard_begin, D, interleave) /
 *                   block_size) <= bt_width, else DCP_ERR_TABLE_TOO_NARROW.
 *
 * The shard of a token and its local index follow the same interleave rule
 * (dcp_shard_of, dcp_local_len).  The workspace is sized by
 * dcp_decode_workspace_size with its D argument = shard_count.
 */
dcp_status_t dcp_mla_decode_partial_local(
    const void* q, int64_t q_stride_tok,
    const void* kv_cache, int32_t num_blocks, int32_t block_size,
    const int32_t* block_table, int32_t bt_width, int64_t bt_stride, int64_t bt_shard_stride,
    const int32_t* seq_lens, const int32_t* query_start_loc,
    int32_t B, int32_t T, int32_t H, int32_t max_seq_len, int32_t max_q_len,
    int32_t D, int32_t interleave, int32_t shard_begin, int32_t shard_count, float scale,
    float* O_part, float* lse_part,
    void* workspace, size_t workspace_bytes,
    int32_t* dev_error, void* stream);

/*
 * The general form of the decode: dcp_mla_decode_partial with every option.
 * The fp8 latent cache and bf16 partials are the pages' next step for the
 * hot path (they halve its two byte streams) ["perf(mla): fuse K3 DCP
 * verification queries", review follow-up: fp8 KV verify plans].
 *
 *   kv_dtype        DCP_KV_BF16: kv_cache bf16 [num_blocks, block_size, 576].
 *                   DCP_KV_FP8_E4M3: kv_cache uint8 codes [num_blocks,
 *                   block_size, 576] and kv_scale fp32 [num_blocks,
 *                   block_size] (required, else DCP_ERR_INVALID_ARG); the
 *                   latent value of a slot is code x scale.  Other values:
 *                   DCP_ERR_UNSUPPORTED_DTYPE.  The tensor-core kernel
 *                   (H <= 128) widens each code x scale to bf16 on its way
 *                   into shared memory (the fp32 product, rounded to
 *                   nearest even): exact when the scale is a power of two,
 *                   else one bf16 rounding of each latent value, as a bf16
 *                   cache holds them.  The CUDA-core kernel applies the
 *                   scale in fp32 to the dot products and the PV weights.
 *   per_shard_tables, bt_shard_stride, shard_begin, shard_count
 *                   0: one table row per request ([B, bt_width]); 1:
 *                   per-shard tables as for dcp_mla_decode_partial_local.
 *                   Either way the call computes shards [shard_begin,
 *                   shard_begin + shard_count) of D.
 *   O_part, o_dtype fp32 or bf16 (round to nearest even) [shard_count, T,
 *                   H, 512]; lse_part stays fp32.  With bf16 the split-KV
 *                   partials in the workspace are bf16 too.
 * Everything else as for dcp_mla_decode_partial.
 */
dcp_status_t dcp_mla_decode_partial_v2(
    const void* q, int64_t q_stride_tok,
    const void* kv_cache, dcp_kv_dtype_t kv_dtype, const float* kv_scale,
    int32_t num_blocks, int32_t block_size,
    const int32_t* block_table, int32_t bt_width, int64_t bt_stride,
    int32_t per_shard_tables, int64_t bt_shard_stride, int32_t shard_begin, int32_t shard_count,
    const int32_t* seq_lens, const int32_t* query_start_loc,
    int32_t B, int32_t T, int32_t H, int32_t max_seq_len, int32_t max_q_len,
    int32_t D, int32_t interleave, float scale,
    void* O_part, dcp_dtype_t o_dtype, float* lse_part,
    void* workspace, size_t workspace_bytes,
    int32_t* dev_error, void* stream);

/*
 * dcp_lse_combine over partials in fp32 or bf16 (part_dtype), e.g. those of
 * dcp_mla_decode_partial_v2 with o_dtype = DCP_DTYPE_BF16.  Everything else
 * as for dcp_lse_combine; an unsupported part_dtype returns
 * DCP_ERR_UNSUPPORTED_DTYPE.
 */
dcp_status_t dcp_lse_combine_v2(
    const void* O_part, dcp_dtype_t part_dtype, const float* lse_part,
    const int32_t* seq_lens, const int32_t* query_start_loc,
    int32_t B, int32_t T, int32_t H, int32_t D,
    void* out, dcp_dtype_t out_dtype, float* out_lse, void* stream);

/*
 * The decode step before attention, fused into one launch ["[Kimi-K3] DCP
 * support" summary on prhub.com.cn, key snippet "Decode: latent multi-query
 * attention": _decode_concat_cache builds the decode query and writes this
 * step's latent rows into the paged cache before forward_mqa, so the decode
 * call sees the new tokens (seq_lens count them)].  The optional RoPE of the
 * snippet (rope_positions = None) is not applied: the rope parts are taken as
 * given.
 *
 * For every token t < T and head h < H:
 *   q_out[t, h, 0:512]   = ql_nope[t, h, :]
 *   q_out[t, h, 512:576] = q_pe[t, h, :]
 * and, when 0 <= slot_mapping[t] < num_slots:
 *   kv_cache[slot_mapping[t], 0:512]   = kv_c[t, :]
 *   kv_cache[slot_mapping[t], 512:576] = k_pe[t, :]
 * slot_mapping[t] = block * block_size + offset is the token's cache row.  A
 * negative slot is not written: a padding token, or (with per-rank caches) a
 * token another DCP rank owns.  A slot >= num_slots is not written either and
 * sets DCP_DEVERR_BAD_BLOCK in *dev_error.  Byte copies: bit-exact.
 *
 *   ql_nope      bf16 [T, H, 512]; element (t, h, k) at t * ql_nope_stride_tok +
 *                h * ql_nope_stride_head + k (e.g. the transposed output of the
 *                per-head q_nope x W_UK batched matmul).
 *   q_pe         bf16 [T, H, 64], strides likewise.
 *   kv_c, k_pe   bf16 [T, 512] and [T, 64], rows kv_c_stride_tok /
 *                k_pe_stride_tok apart.
 *   slot_mapping int64 [T], device.
 *   q_out        bf16 [T, H, 576], heads dense, rows q_out_stride_tok apart
 *                (>= H * 576); must not overlap any input.
 *   kv_cache     bf16 [num_slots, 576] (num_blocks * block_size rows); two
 *                tokens must not share a slot.
 * Every pointer is 16-byte aligned and every stride a multiple of 8
 * elements, else DCP_ERR_MISALIGNED.  T == 0 returns DCP_OK without
 * launching anything.
 */
dcp_status_t dcp_decode_concat_cache(
    const void* ql_nope, int64_t ql_nope_stride_tok, int64_t ql_nope_stride_head,
    const void* q_pe, int64_t q_pe_stride_tok, int64_t q_pe_stride_head,
    const void* kv_c, int64_t kv_c_stride_tok,
    const void* k_pe, int64_t k_pe_stride_tok,
    const int64_t* slot_mapping, int32_t T, int32_t H,
    void* q_out, int64_t q_out_stride_tok,
    void* kv_cache, int64_t num_slots,
    int32_t* dev_error, void* stream);

/*
 * dcp_mla_decode_partial without a workspace argument, for callers that
 * cannot allocate device memory (their memory is owned and fully reserved by
 * a host framework, or they are plugins handed only their inputs and
 * outputs).  The pages have no counterpart: it is a packaging of the same
 * decode.
 *
 * Same arguments, results and errors as dcp_mla_decode_partial, except that
 * the split-KV scratch comes from a 24 MiB array inside the library (held on
 * every device that loads it, until the process exits).  A call whose split
 * plan needs more than 24 MiB (dcp_decode_workspace_size) returns
 * DCP_ERR_WORKSPACE_TOO_SMALL without launching; H <= 128 always fits on a
 * GB300.  The first call on a device looks up the array's device address, so
 * make it before capturing a stream on that device.  All calls share the
 * array and it keeps the last call's contents (nothing in it needs to start
 * at zero); calls whose kernels overlap on the GPU race on it, so order them
 * on one stream or with events.  Allocates nothing.
 */
dcp_status_t dcp_mla_decode_partial_noalloc(
    const void* q, int64_t q_stride_tok,
    const void* kv_cache, int32_t num_blocks, int32_t block_size,
    const int32_t* block_table, int32_t bt_width, int64_t bt_stride,
    const int32_t* seq_lens, const int32_t* query_start_loc,
    int32_t B, int32_t T, int32_t H, int32_t max_seq_len, int32_t max_q_len,
    int32_t D, int32_t interleave, float scale,
    float* O_part, float* lse_part,
    int32_t* dev_error, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DCP_H_ */
