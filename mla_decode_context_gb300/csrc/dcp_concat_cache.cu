// The decode step before attention, in one launch: the decode query
// q = [ql_nope | q_pe] (576 bf16 per head) and the write of this step's latent
// rows [kv_c | k_pe] into the paged cache at slot_mapping ("[Kimi-K3] DCP
// support" summary on prhub.com.cn, key snippet "Decode: latent multi-query
// attention": _decode_concat_cache runs before forward_mqa, so the decode
// sees the new tokens).  Byte copies only (bit-exact), in 16-byte units.
//
// One CTA per token: its eight warps copy the token's H query heads (72
// 16-byte units per head: 64 of ql_nope, then 8 of q_pe), and warp 0 also
// copies its cache row when the slot is set.  A negative slot is not written
// (a padding token, or a token another DCP rank owns); a slot past the cache
// is not written either and sets DCP_DEVERR_BAD_BLOCK.
#include "dcp_kernels.h"

namespace dcp {
namespace {

constexpr int kThreads = 256;
constexpr int kUnitsNope = kLatent * 2 / 16;  // 64 16-byte units of ql_nope / kv_c
constexpr int kUnitsRope = kRope * 2 / 16;    // 8 of q_pe / k_pe
constexpr int kUnitsRow = kUnitsNope + kUnitsRope;

__device__ __forceinline__ uint4 ld_nc(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

__global__ void __launch_bounds__(kThreads) concat_cache_kernel(ConcatCacheArgs a) {
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned char* nope = reinterpret_cast<const unsigned char*>(a.ql_nope) + 2 * t * a.ql_nope_stride_tok;
  const unsigned char* pe = reinterpret_cast<const unsigned char*>(a.q_pe) + 2 * t * a.q_pe_stride_tok;
  unsigned char* qo = reinterpret_cast<unsigned char*>(a.q_out) + 2 * t * a.q_out_stride_tok;
  for (int h = warp; h < a.H; h += kThreads / 32) {
    const unsigned char* n = nope + 2 * h * a.ql_nope_stride_head;
    const unsigned char* p = pe + 2 * h * a.q_pe_stride_head;
    uint4* dst = reinterpret_cast<uint4*>(qo + 2 * h * kKDim);
    for (int u = lane; u < kUnitsRow; u += 32) dst[u] = u < kUnitsNope ? ld_nc(n + 16 * u) : ld_nc(p + 16 * (u - kUnitsNope));
  }
  if (warp == 0) {
    const int64_t slot = __ldg(a.slot_mapping + t);
    if (slot >= a.num_slots) {
      if (lane == 0 && a.dev_error) atomicOr(a.dev_error, DCP_DEVERR_BAD_BLOCK);
    } else if (slot >= 0) {
      const unsigned char* c = reinterpret_cast<const unsigned char*>(a.kv_c) + 2 * t * a.kv_c_stride_tok;
      const unsigned char* k = reinterpret_cast<const unsigned char*>(a.k_pe) + 2 * t * a.k_pe_stride_tok;
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(a.kv_cache) + slot * (2 * kKDim));
      for (int u = lane; u < kUnitsRow; u += 32) dst[u] = u < kUnitsNope ? ld_nc(c + 16 * u) : ld_nc(k + 16 * (u - kUnitsNope));
    }
  }
}

}  // namespace

cudaError_t launch_concat_cache(const ConcatCacheArgs& a, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  concat_cache_kernel<<<a.T, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace dcp
