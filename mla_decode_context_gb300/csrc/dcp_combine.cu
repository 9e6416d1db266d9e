// LSE-weighted combine / split merge: a vectorised, coalesced streaming
// reduction (no tensor cores; HBM-bound).
//
// One warp owns one (row, head) pair.  Lane d < nsrc reads source d's LSE;
// the live set E = {d : lse_d != -inf} is a warp ballot, so the partial
// output of a masked source is never loaded [spec formula; the
// "[Kimi-K3] DCP support" summary on prhub.com.cn, implementation step 4:
// -inf at the source, zero-weight sources skipped by the consumer].
// Weights are exp2(lse_d * log2 e - M) with M the maximum over E; the 512
// outputs are spread over the warp as four 16-byte loads per lane and
// source, so every load instruction reads 512 contiguous bytes.
#include "dcp_kernels.h"

#include <cmath>

namespace dcp {
namespace {

constexpr int kWarpsPerCta = 8;
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

template <typename OutT, bool kRowMask>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
lse_merge_kernel(const float* __restrict__ O_src, const float* __restrict__ lse_src,
                 int64_t o_stride, int64_t lse_stride, int nsrc, int64_t npairs, int32_t H,
                 const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ qsl, int32_t B,
                 OutT* __restrict__ out, float* out_lse) {
  const int lane = threadIdx.x & 31;
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  if (pair >= npairs) return;
  OutT* dst = out + pair * kLatent;

  bool pad = false;
  if (kRowMask) pad = row_is_padding(seq_lens, qsl, B, static_cast<int32_t>(pair / H));
  if (!pad) {
    // out_lse may alias lse_src's source-0 slice: all reads of this pair's
    // LSEs happen here, before the single write below.
    const float l = lane < nsrc ? __ldg(lse_src + lane * lse_stride + pair) : -INFINITY;
    const bool live = l != -INFINITY;
    unsigned live_mask = __ballot_sync(kFull, live);
    if (live_mask) {
      const float l2 = live ? l * kLog2e : -INFINITY;
      const float M = warp_max(l2);
      const float w = live ? exp2f(l2 - M) : 0.f;
      const float den = warp_sum(w);
      float4 acc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      while (live_mask) {
        const int d = __ffs(live_mask) - 1;
        live_mask &= live_mask - 1;
        const float wd = __shfl_sync(kFull, w, d);
        const float4* src = reinterpret_cast<const float4*>(O_src + d * o_stride + pair * kLatent);
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = __ldcs(src + lane + 32 * k);  // streamed once
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[k].x = fmaf(wd, v[k].x, acc[k].x);
          acc[k].y = fmaf(wd, v[k].y, acc[k].y);
          acc[k].z = fmaf(wd, v[k].z, acc[k].z);
          acc[k].w = fmaf(wd, v[k].w, acc[k].w);
        }
      }
      const float inv = 1.f / den;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float4 o = acc[k];
        o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
        store4(dst + 4 * lane + 128 * k, o);
      }
      if (lane == 0) out_lse[pair] = (M + log2f(den)) * kLn2;
      return;
    }
  }
  // padding row, or no live source: zeros and -inf, nothing else read
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 4; ++k) store4(dst + 4 * lane + 128 * k, z);
  if (lane == 0) out_lse[pair] = -INFINITY;
}

template <typename OutT, bool kRowMask>
cudaError_t launch(const float* O_src, const float* lse_src, int64_t o_stride, int64_t lse_stride,
                   int nsrc, int64_t npairs, int32_t H, const int32_t* seq_lens, const int32_t* qsl,
                   int32_t B, OutT* out, float* out_lse, cudaStream_t st) {
  if (npairs <= 0) return cudaSuccess;
  const int64_t grid = (npairs + kWarpsPerCta - 1) / kWarpsPerCta;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  lse_merge_kernel<OutT, kRowMask><<<static_cast<unsigned>(grid), kWarpsPerCta * 32, 0, st>>>(
      O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H, seq_lens, qsl, B, out, out_lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lse_merge_bf16(const float* O_src, const float* lse_src, int64_t o_stride,
                                  int64_t lse_stride, int nsrc, int64_t npairs, int32_t H,
                                  const int32_t* seq_lens, const int32_t* qsl, int32_t B,
                                  __nv_bfloat16* out, float* out_lse, cudaStream_t st) {
  return launch<__nv_bfloat16, true>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H,
                                     seq_lens, qsl, B, out, out_lse, st);
}

cudaError_t launch_lse_merge_f32(const float* O_src, const float* lse_src, int64_t o_stride,
                                 int64_t lse_stride, int nsrc, int64_t npairs, int32_t H,
                                 const int32_t* seq_lens, const int32_t* qsl, int32_t B,
                                 bool row_mask, float* out, float* out_lse, cudaStream_t st) {
  if (row_mask)
    return launch<float, true>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H, seq_lens,
                               qsl, B, out, out_lse, st);
  return launch<float, false>(O_src, lse_src, o_stride, lse_stride, nsrc, npairs, H, seq_lens,
                              qsl, B, out, out_lse, st);
}

}  // namespace dcp
