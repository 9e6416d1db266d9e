// Reference split-KV MLA decode on the CUDA cores (fp32 FMA).
//
// Handles every geometry the C ABI accepts (any H, block size, D,
// interleave).  One CTA = (row r, shard d, split s, group of 8 heads); one
// warp per head.  A tile of 32 shard tokens is staged in shared memory (bf16,
// rows padded to 1168 bytes so that lane = token reads are bank-conflict
// free); lane t computes token t's 576-wide score, the warp runs an online
// softmax in base 2, then every lane accumulates 16 of the 512 value dims.
// Tokens outside the shard range or behind a bad block id are staged as
// zeros and masked to weight 0 by selection (never NaN * 0).  An FP8 E4M3
// cache is staged as its codes (576 bytes a row) with each row's scale, and
// widened on use (exactly: every E4M3 value is a half) before the scale is
// applied; partial outputs may be written in bf16.
#include "dcp_kernels.h"

#include <cuda_fp8.h>
#include <cmath>
#include <mutex>

namespace dcp {
namespace {

constexpr int kHeadsPerCta = 8;
constexpr int kThreads = kHeadsPerCta * 32;
constexpr int kTile = 32;
constexpr int kRowBytes = kKDim * 2 + 16;  // 1168: padded smem row
constexpr int kChunks = kKDim * 2 / 16;    // 72 16-byte chunks per latent row
constexpr unsigned kFull = 0xffffffffu;

struct alignas(16) Smem {
  unsigned char kv[kTile][kRowBytes];
  float q[kHeadsPerCta][kKDim];
  int64_t phys[kTile];
  float kv_scale[kTile];
};

// four / two E4M3 codes widened to fp32 (exact)
__device__ __forceinline__ float2 fp8x2_to_float2(uint16_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__global__ void __launch_bounds__(kThreads)
decode_simt_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = (a.H + kHeadsPerCta - 1) / kHeadsPerCta;
  const int hg = blockIdx.x % groups;
  const int r = blockIdx.x / groups;
  const int h = hg * kHeadsPerCta + warp;
  const int d = a.d0 + static_cast<int>(blockIdx.y) / a.plan.splits;  // shard (of D)
  const int s = blockIdx.y % a.plan.splits;
  const bool head_ok = h < a.H;

  const int64_t dst_pair = ((static_cast<int64_t>(s) * a.Dn + (d - a.d0)) * a.T + r) * a.H + h;
  const bool fp8 = a.kv_fp8 != 0;

  const RowInfo ri = resolve_row(a.seq_lens, a.qsl, a.B, r, a.max_seq_len, a.max_q_len);
  if (ri.err && threadIdx.x == 0 && hg == 0 && blockIdx.y == 0 && a.dev_error)
    atomicOr(a.dev_error, static_cast<int32_t>(ri.err));
  const int32_t n_local = ri.padding ? 0 : local_len(ri.L, d, a.D, a.I);
  const int32_t lo = s * a.plan.chunk;
  const int32_t hi = min(n_local, lo + a.plan.chunk);

  float m = -INFINITY, l = 0.f;  // running max (log2 domain) and sum
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;

  if (lo < hi) {
    // this warp's query head, widened to fp32
    for (int i = threadIdx.x; i < kHeadsPerCta * kKDim; i += kThreads) {
      const int hh = hg * kHeadsPerCta + i / kKDim;
      float v = 0.f;
      if (hh < a.H) {
        const __nv_bfloat16* qp = a.q + static_cast<int64_t>(r) * a.q_stride_tok + static_cast<int64_t>(hh) * kKDim;
        v = __bfloat162float(qp[i % kKDim]);
      }
      sm.q[i / kKDim][i % kKDim] = v;
    }
    const float sl2 = a.scale * kLog2e;
    const int32_t* trow = a.block_table + static_cast<int64_t>(ri.b) * a.bt_stride +
                          (a.local_tables ? static_cast<int64_t>(d - a.d0) * a.bt_shard_stride : 0);

    for (int32_t t0 = lo; t0 < hi; t0 += kTile) {
      __syncthreads();  // previous tile fully consumed (and q staged)
      if (threadIdx.x < kTile) {
        const int32_t j = t0 + threadIdx.x;
        int64_t phys = -1;
        if (j < hi) {
          // table index: the shard token's position, or its local index (per-shard layout)
          const int64_t p = a.local_tables ? j : local_to_global(j, d, a.D, a.I);
          const int32_t blk = __ldg(trow + p / a.block_size);
          if (blk >= 0 && blk < a.num_blocks)
            phys = static_cast<int64_t>(blk) * a.block_size + p % a.block_size;
          else if (a.dev_error)
            atomicOr(a.dev_error, DCP_DEVERR_BAD_BLOCK);
        }
        sm.phys[threadIdx.x] = phys;
        sm.kv_scale[threadIdx.x] = fp8 && phys >= 0 ? __ldg(a.kv_scale + phys) : 1.f;
      }
      __syncthreads();
      // 16-byte units of a row: 72 (bf16) or 36 (fp8 codes)
      const int units = fp8 ? kChunks / 2 : kChunks;
      const int row_bytes = fp8 ? kKDim : 2 * kKDim;
      for (int c = threadIdx.x; c < kTile * units; c += kThreads) {
        const int row = c / units, col = c % units;
        const int64_t phys = sm.phys[row];
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (phys >= 0)
          v = __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(a.kv) + phys * row_bytes) + col);
        *reinterpret_cast<uint4*>(&sm.kv[row][col * 16]) = v;
      }
      __syncthreads();
      if (!head_ok) continue;

      // scores: lane = token
      float sc = 0.f;
      const uint4* krow = reinterpret_cast<const uint4*>(&sm.kv[lane][0]);
      const float4* qv = reinterpret_cast<const float4*>(&sm.q[warp][0]);
      if (!fp8) {
#pragma unroll 4
        for (int c = 0; c < kChunks; ++c) {
          const uint4 k = krow[c];
          const float4 q0 = qv[2 * c], q1 = qv[2 * c + 1];
          sc = fmaf(q0.x, bf16lo(k.x), sc); sc = fmaf(q0.y, bf16hi(k.x), sc);
          sc = fmaf(q0.z, bf16lo(k.y), sc); sc = fmaf(q0.w, bf16hi(k.y), sc);
          sc = fmaf(q1.x, bf16lo(k.z), sc); sc = fmaf(q1.y, bf16hi(k.z), sc);
          sc = fmaf(q1.z, bf16lo(k.w), sc); sc = fmaf(q1.w, bf16hi(k.w), sc);
        }
      } else {
        // 16 codes per unit; the row's scale multiplies the dot product
#pragma unroll 2
        for (int c = 0; c < kChunks / 2; ++c) {
          const uint4 k = krow[c];
          const uint32_t w[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 qq = qv[4 * c + i];
            const float2 lo = fp8x2_to_float2(static_cast<uint16_t>(w[i] & 0xffffu));
            const float2 hi = fp8x2_to_float2(static_cast<uint16_t>(w[i] >> 16));
            sc = fmaf(qq.x, lo.x, sc); sc = fmaf(qq.y, lo.y, sc);
            sc = fmaf(qq.z, hi.x, sc); sc = fmaf(qq.w, hi.y, sc);
          }
        }
        sc *= sm.kv_scale[lane];
      }
      const bool valid = sm.phys[lane] >= 0;
      const float s2 = valid ? sc * sl2 : -INFINITY;
      float tmax = s2;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o));
      const float m_new = fmaxf(m, tmax);
      if (m_new == -INFINITY) continue;  // nothing valid yet
      const float alpha = exp2f(m - m_new);
      const float p = valid ? exp2f(s2 - m_new) : 0.f;
      float psum = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(kFull, psum, o);
      l = l * alpha + psum;
      m = m_new;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] *= alpha;
      // values: lane owns dims 4*lane + 128*k .. +3
      for (int t = 0; t < kTile; ++t) {
        const float pt = __shfl_sync(kFull, p, t);
        if (pt == 0.f) continue;  // warp-uniform
        if (!fp8) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint2 v = *reinterpret_cast<const uint2*>(&sm.kv[t][(4 * lane + 128 * k) * 2]);
            acc[4 * k + 0] = fmaf(pt, bf16lo(v.x), acc[4 * k + 0]);
            acc[4 * k + 1] = fmaf(pt, bf16hi(v.x), acc[4 * k + 1]);
            acc[4 * k + 2] = fmaf(pt, bf16lo(v.y), acc[4 * k + 2]);
            acc[4 * k + 3] = fmaf(pt, bf16hi(v.y), acc[4 * k + 3]);
          }
        } else {
          const float ps = pt * sm.kv_scale[t];  // weight x the row's scale
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t v = *reinterpret_cast<const uint32_t*>(&sm.kv[t][4 * lane + 128 * k]);
            const float2 lo = fp8x2_to_float2(static_cast<uint16_t>(v & 0xffffu));
            const float2 hi = fp8x2_to_float2(static_cast<uint16_t>(v >> 16));
            acc[4 * k + 0] = fmaf(ps, lo.x, acc[4 * k + 0]);
            acc[4 * k + 1] = fmaf(ps, lo.y, acc[4 * k + 1]);
            acc[4 * k + 2] = fmaf(ps, hi.x, acc[4 * k + 2]);
            acc[4 * k + 3] = fmaf(ps, hi.y, acc[4 * k + 3]);
          }
        }
      }
    }
  }
  if (!head_ok) return;
  // empty shard / split, or padding row: masked at the source (0 / -inf)
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 v = make_float4(acc[4 * k] * inv, acc[4 * k + 1] * inv, acc[4 * k + 2] * inv, acc[4 * k + 3] * inv);
    if (!a.o_bf16) {
      *reinterpret_cast<float4*>(static_cast<float*>(a.O_dst) + dst_pair * kLatent + 4 * lane + 128 * k) = v;
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.O_dst) + dst_pair * kLatent + 4 * lane + 128 * k) =
          make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    }
  }
  if (lane == 0) a.lse_dst[dst_pair] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(Smem);
  // shared-memory opt-in once per device (not per launch: launches may be
  // captured into a CUDA graph)
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      done[dev] = true;
    }
  }
  const int64_t gx = static_cast<int64_t>((a.H + kHeadsPerCta - 1) / kHeadsPerCta) * a.T;
  const int64_t gy = static_cast<int64_t>(a.Dn) * a.plan.splits;
  if (gx > 0x7fffffffLL || gy > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  decode_simt_kernel<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace dcp
