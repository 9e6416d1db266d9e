// LSE-weighted combine / split merge: a streaming reduction over nsrc
// partials (no tensor cores; HBM/L2-bound, and latency-bound when there are
// few (row, head) pairs).
//
// kQ warps own one (row, head) pair, each a 512 / kQ-column share of its
// output, 8 / kQ pairs per CTA.  Lane d of each warp reads source d's LSE,
// the live set E = {d : lse_d != -inf} is a warp ballot, and the weights
// exp2(lse_d log2 e - M) (M = max over E) are warp reductions; a masked
// source adds nothing to the sum ["[Kimi-K3] DCP support" summary on
// prhub.com.cn, implementation step 4: -inf at the source, zero-weight
// sources skipped by the consumer].  Lane t owns kF = 4 / kQ float4 columns
// of each source (columns 4t + 128k of its warp's share), so every load and
// store of a warp is a contiguous 512-byte access.  Two ways to load:
//   batched (kEarly = false): after the weights, the live sources only,
//     kBatch at a time.  A masked source's partial is never read.  The
//     combine takes this way with one warp per pair when there are many
//     pairs, so that many pairs per SM keep enough bytes in flight.
//   early (kEarly = true): every source's partial is loaded before the
//     weights are known (one memory round trip in all) and the sum takes the
//     live ones only, so the bytes of a masked source (NaN or anything) are
//     read but never used.  The split merge (up to 16 splits) and the
//     combine of few pairs take this way: two warps per pair up to 8 or 12
//     sources, four warps up to 16; a thread holds at most 96 loaded
//     registers and two 256-thread CTAs fit on an SM.
// Both ways sum the live sources in increasing index order with the same
// weights, so they give bit-identical results and every result is
// deterministic.  The kernel waits on the grid it depends on (programmatic
// dependent launch) only after its launch, so its launch overlaps the tail of
// the kernel that produced its inputs.
#include "dcp_kernels.h"

#include <cmath>

namespace dcp {
namespace {

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);  // round to nearest even
  __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

// 16-byte (fp32) or 8-byte (bf16) streaming load of four partial-output
// columns, widened to fp32
__device__ __forceinline__ float4 load4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void fma4(float4& acc, float w, const float4& v) {
  acc.x = fmaf(w, v.x, acc.x);
  acc.y = fmaf(w, v.y, acc.y);
  acc.z = fmaf(w, v.z, acc.z);
  acc.w = fmaf(w, v.w, acc.w);
}

// kQ warps per pair; the early way loads all nsrc <= kBatch sources at once,
// the batched way kBatch live sources at a time
template <typename InT, typename OutT, bool kRowMask, bool kEarly, int kQ, int kBatch>
__global__ void __launch_bounds__(kThreads, (!kEarly && kBatch <= 2) ? 4 : 2)
lse_merge_kernel(const InT* __restrict__ O_src, const float* __restrict__ lse_src,
                 int64_t o_stride, int64_t lse_stride, int nsrc, int64_t npairs, int32_t H,
                 const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ qsl, int32_t B,
                 OutT* __restrict__ out, float* out_lse) {
  constexpr int kF = 4 / kQ;                     // float4 columns per lane per source
  constexpr int kPairs = kThreads / 32 / kQ;     // pairs per CTA
  asm volatile("griddepcontrol.wait;" ::: "memory");  // inputs written by the preceding grid
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * kPairs + w / kQ;
  const int share = w % kQ;
  const bool has = pair < npairs;
  const InT* src = O_src + pair * kLatent + share * (kLatent / kQ) + 4 * lane;

  float4 pre[kEarly ? kBatch : 1][kF];
  if (kEarly && has) {
#pragma unroll
    for (int k = 0; k < (kEarly ? kBatch : 1); ++k)
      if (k < nsrc) {
#pragma unroll
        for (int f = 0; f < kF; ++f) pre[k][f] = load4(src + k * o_stride + 128 * f);
      }
  }

  // the LSE loads go out together with the row's padding test (a padding
  // row's LSEs are read but ignored)
  const float l_raw = has && lane < nsrc ? __ldg(lse_src + lane * lse_stride + pair) : -INFINITY;
  bool pad = false;
  if (kRowMask && has) pad = row_is_padding(seq_lens, qsl, B, static_cast<int32_t>(pair / H));
  const float l = pad ? -INFINITY : l_raw;
  const bool live = l != -INFINITY;
  const unsigned live_mask = __ballot_sync(kFull, live);
  const float l2 = live ? l * kLog2e : -INFINITY;
  const float M = live_mask ? warp_max(l2) : 0.f;
  const float wt = live ? exp2f(l2 - M) : 0.f;
  const float den = warp_sum(wt);
  // out_lse may alias lse_src's source-0 slice: every warp of a pair has read
  // its LSEs before the single write below (with one warp per pair, the
  // ballot above already orders them: l_raw is consumed before it)
  if (kQ > 1) __syncthreads();
  if (!has) return;
  if (share == 0 && lane == 0) out_lse[pair] = live_mask ? (M + log2f(den)) * kLn2 : -INFINITY;

  float4 acc[kF];
#pragma unroll
  for (int f = 0; f < kF; ++f) acc[f] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (kEarly) {
    // the live sources in increasing index (a padding row has none)
#pragma unroll
    for (int k = 0; k < (kEarly ? kBatch : 1); ++k)
      if (k < nsrc && ((live_mask >> k) & 1u)) {
        const float wd = __shfl_sync(kFull, wt, k);
#pragma unroll
        for (int f = 0; f < kF; ++f) fma4(acc[f], wd, pre[k][f]);
      }
  } else {
    unsigned m = live_mask;  // padding row or no live source: m == 0, so zeros
    while (m) {
      int ds[kBatch];
      int n = 0;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        ds[i] = m ? __ffs(m) - 1 : 0;
        n += m ? 1 : 0;
        m &= m - 1;
      }
      float4 v[kBatch][kF];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        if (i < n) {
#pragma unroll
          for (int f = 0; f < kF; ++f) v[i][f] = load4(src + ds[i] * o_stride + 128 * f);
        }
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        if (i < n) {
          const float wd = __shfl_sync(kFull, wt, ds[i]);
#pragma unroll
          for (int f = 0; f < kF; ++f) fma4(acc[f], wd, v[i][f]);
        }
    }
  }
  const float inv = live_mask ? 1.f / den : 0.f;
  OutT* dst = out + pair * kLatent + share * (kLatent / kQ) + 4 * lane;
#pragma unroll
  for (int f = 0; f < kF; ++f)
    store4(dst + 128 * f, make_float4(acc[f].x * inv, acc[f].y * inv, acc[f].z * inv, acc[f].w * inv));
}

template <typename InT, typename OutT, bool kRowMask, bool kEarly, int kQ, int kBatch>
cudaError_t launch_batch(const InT* O_src, const float* lse_src, int64_t o_stride, int64_t lse_stride, int nsrc,
                         int64_t npairs, int32_t H, const int32_t* seq_lens, const int32_t* qsl, int32_t B,
                         OutT* out, float* out_lse, cudaStream_t st) {
  constexpr int kPairs = kThreads / 32 / kQ;
  const int64_t ctas = (npairs + kPairs - 1) / kPairs;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lse_merge_kernel<InT, OutT, kRowMask, kEarly, kQ, kBatch>, O_src, lse_src,
                            o_stride, lse_stride, nsrc, npairs, H, seq_lens, qsl, B, out, out_lse);
}

// Below this many pairs one warp per pair leaves most SMs idle (eight pairs
// per 256-thread CTA), and the combine loads early instead.
constexpr int64_t kFewPairs = 2048;

// The early way: all sources at once, two warps per pair up to 12 sources,
// four up to 16; past 16 the batched way with four warps per pair.
template <typename InT, typename OutT, bool kRowMask>
cudaError_t launch_early(const InT* O_src, const float* lse_src, int64_t o_stride, int64_t lse_stride, int nsrc,
                         int64_t npairs, int32_t H, const int32_t* seq_lens, const int32_t* qsl, int32_t B,
                         OutT* out, float* out_lse, cudaStream_t st) {
  if (nsrc <= 8)
    return launch_batch<InT, OutT, kRowMask, true, 2, 8>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H,
                                                         seq_lens, qsl, B, out, out_lse, st);
  if (nsrc <= 12)
    return launch_batch<InT, OutT, kRowMask, true, 2, 12>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H,
                                                          seq_lens, qsl, B, out, out_lse, st);
  if (nsrc <= 16)
    return launch_batch<InT, OutT, kRowMask, true, 4, 16>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H,
                                                          seq_lens, qsl, B, out, out_lse, st);
  return launch_batch<InT, OutT, kRowMask, false, 4, 16>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H,
                                                         seq_lens, qsl, B, out, out_lse, st);
}

// The split merge loads early.  The combine of many pairs (one warp per pair,
// four float4 columns per lane per source) loads two live sources at a time
// when there are at most two, else four: fewer registers for small D leave
// room for more pairs per SM.
template <typename InT, typename OutT, bool kRowMask>
cudaError_t launch(const InT* O_src, const float* lse_src, int64_t o_stride, int64_t lse_stride, int nsrc,
                   int64_t npairs, int32_t H, const int32_t* seq_lens, const int32_t* qsl, int32_t B, OutT* out,
                   float* out_lse, cudaStream_t st) {
  if (npairs <= 0) return cudaSuccess;
  if (!kRowMask || npairs < kFewPairs)
    return launch_early<InT, OutT, kRowMask>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H, seq_lens, qsl,
                                             B, out, out_lse, st);
  if constexpr (kRowMask) {
    if (nsrc <= 2)
      return launch_batch<InT, OutT, kRowMask, false, 1, 2>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H,
                                                            seq_lens, qsl, B, out, out_lse, st);
    return launch_batch<InT, OutT, kRowMask, false, 1, 4>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H,
                                                          seq_lens, qsl, B, out, out_lse, st);
  }
  return cudaSuccess;
}

template <typename InT>
cudaError_t launch_in(const InT* O_src, const float* lse_src, int64_t o_stride, int64_t lse_stride, int nsrc,
                      int64_t npairs, int32_t H, const int32_t* seq_lens, const int32_t* qsl, int32_t B,
                      bool row_mask, void* out, bool out_bf16, float* out_lse, cudaStream_t st) {
  if (row_mask) {
    if (out_bf16)
      return launch<InT, __nv_bfloat16, true>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H, seq_lens, qsl,
                                              B, static_cast<__nv_bfloat16*>(out), out_lse, st);
    return launch<InT, float, true>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H, seq_lens, qsl, B,
                                    static_cast<float*>(out), out_lse, st);
  }
  if (out_bf16)
    return launch<InT, __nv_bfloat16, false>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H, seq_lens, qsl,
                                             B, static_cast<__nv_bfloat16*>(out), out_lse, st);
  return launch<InT, float, false>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H, seq_lens, qsl, B,
                                   static_cast<float*>(out), out_lse, st);
}

}  // namespace

cudaError_t launch_lse_merge(const void* O_src, bool src_bf16, const float* lse_src, int64_t o_stride,
                             int64_t lse_stride, int nsrc, int64_t npairs, int32_t H, const int32_t* seq_lens,
                             const int32_t* qsl, int32_t B, bool row_mask, void* out, bool out_bf16,
                             float* out_lse, cudaStream_t st) {
  if (src_bf16)
    return launch_in(static_cast<const __nv_bfloat16*>(O_src), lse_src, o_stride, lse_stride, nsrc, npairs, H,
                     seq_lens, qsl, B, row_mask, out, out_bf16, out_lse, st);
  return launch_in(static_cast<const float*>(O_src), lse_src, o_stride, lse_stride, nsrc, npairs, H, seq_lens, qsl,
                   B, row_mask, out, out_bf16, out_lse, st);
}

}  // namespace dcp
