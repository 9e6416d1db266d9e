// LSE-weighted combine / split merge: a streaming reduction over nsrc
// partials (no tensor cores; HBM/L2-bound, and latency-bound when there are
// few (row, head) pairs).
//
// One 128-thread CTA owns one (row, head) pair.  Warp 0 reads the nsrc LSEs
// (lane d: source d), takes the live set E = {d : lse_d != -inf} as a warp
// ballot, and publishes the weights exp2(lse_d log2 e - M) (M = max over E;
// 0 outside E) to shared memory; the partial output of a masked source is
// never loaded ["[Kimi-K3] DCP support" summary on prhub.com.cn,
// implementation step 4: -inf at the source, zero-weight sources skipped by
// the consumer].  Thread t then owns output columns 4t .. 4t+3 and issues
// the 16-byte loads of up to 8 sources at once, so a pair costs one or two
// memory round trips instead of one per source.  The kernel waits on the
// grid it depends on (programmatic dependent launch) only after its launch,
// so its launch overlaps the tail of the kernel that produced its inputs.
#include "dcp_kernels.h"

#include <cmath>

namespace dcp {
namespace {

constexpr int kThreadsPerPair = kLatent / 4;  // one float4 column each
constexpr int kBatch = 8;                     // sources loaded per round trip
constexpr int kAllAtOnce = 16;                // split merge: sources loaded before the weights are known
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
__global__ void __launch_bounds__(kThreadsPerPair)
lse_merge_kernel(const float* __restrict__ O_src, const float* __restrict__ lse_src,
                 int64_t o_stride, int64_t lse_stride, int nsrc, int64_t npairs, int32_t H,
                 const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ qsl, int32_t B,
                 OutT* __restrict__ out, float* out_lse) {
  __shared__ float w_s[32];
  __shared__ float wd_s[32];  // weight by source index (0 if masked)
  __shared__ int32_t live_s[32];
  __shared__ int32_t nlive_s;
  __shared__ float inv_s;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // inputs written by the preceding grid
  const int t = threadIdx.x, lane = t & 31;
  const int64_t pair = blockIdx.x;
  OutT* dst = out + pair * kLatent + 4 * t;

  // Split merge (no row mask): every source is a split partial that the
  // decode wrote, finite even when its split held no token (zeros, LSE
  // -inf).  So the partials can be loaded while the weights are still being
  // worked out: one memory round trip instead of two or three.
  float4 v_all[kAllAtOnce];
  const bool all_at_once = !kRowMask && nsrc <= kAllAtOnce;
  if (all_at_once) {
#pragma unroll
    for (int k = 0; k < kAllAtOnce; ++k)
      if (k < nsrc) v_all[k] = __ldcs(reinterpret_cast<const float4*>(O_src + k * o_stride + pair * kLatent) + t);
  }

  if (t < 32) {
    bool pad = false;
    if (kRowMask) pad = row_is_padding(seq_lens, qsl, B, static_cast<int32_t>(pair / H));
    // out_lse may alias lse_src's source-0 slice: every read of this pair's
    // LSEs happens here, before the single write below.
    const float l = !pad && lane < nsrc ? __ldg(lse_src + lane * lse_stride + pair) : -INFINITY;
    const bool live = l != -INFINITY;
    const unsigned live_mask = __ballot_sync(kFull, live);
    const float l2 = live ? l * kLog2e : -INFINITY;
    const float M = live_mask ? warp_max(l2) : 0.f;
    const float w = live ? exp2f(l2 - M) : 0.f;
    const float den = warp_sum(w);
    if (live) {
      const int k = __popc(live_mask & ((1u << lane) - 1u));  // rank among the live sources
      live_s[k] = lane;
      w_s[k] = w;
    }
    wd_s[lane] = w;
    if (lane == 0) {
      nlive_s = __popc(live_mask);
      inv_s = live_mask ? 1.f / den : 0.f;
      out_lse[pair] = live_mask ? (M + log2f(den)) * kLn2 : -INFINITY;
    }
  }
  __syncthreads();
  const int n = nlive_s;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (all_at_once) {
    // sources in increasing index, as below; a masked one adds 0 * finite
#pragma unroll
    for (int k = 0; k < kAllAtOnce; ++k)
      if (k < nsrc) {
        const float wd = wd_s[k];
        acc.x = fmaf(wd, v_all[k].x, acc.x);
        acc.y = fmaf(wd, v_all[k].y, acc.y);
        acc.z = fmaf(wd, v_all[k].z, acc.z);
        acc.w = fmaf(wd, v_all[k].w, acc.w);
      }
  }
  for (int k0 = 0; !all_at_once && k0 < n; k0 += kBatch) {
    float4 v[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      if (k0 + k < n)
        v[k] = __ldcs(reinterpret_cast<const float4*>(O_src + live_s[k0 + k] * o_stride + pair * kLatent) + t);
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      if (k0 + k < n) {
        const float wd = w_s[k0 + k];
        acc.x = fmaf(wd, v[k].x, acc.x);
        acc.y = fmaf(wd, v[k].y, acc.y);
        acc.z = fmaf(wd, v[k].z, acc.z);
        acc.w = fmaf(wd, v[k].w, acc.w);
      }
  }
  // padding row or no live source: n == 0, inv == 0, so zeros
  const float inv = inv_s;
  acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
  store4(dst, acc);
}

template <typename OutT, bool kRowMask>
cudaError_t launch(const float* O_src, const float* lse_src, int64_t o_stride, int64_t lse_stride,
                   int nsrc, int64_t npairs, int32_t H, const int32_t* seq_lens, const int32_t* qsl,
                   int32_t B, OutT* out, float* out_lse, cudaStream_t st) {
  if (npairs <= 0) return cudaSuccess;
  if (npairs > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(npairs));
  cfg.blockDim = dim3(kThreadsPerPair);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lse_merge_kernel<OutT, kRowMask>, O_src, lse_src, o_stride, lse_stride, nsrc,
                            npairs, H, seq_lens, qsl, B, out, out_lse);
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
