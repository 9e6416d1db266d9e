// Probe: tcgen05.mma kind::f16 issue/execution rate, M=128, K=16, bf16, fp32
// accumulators, A from TMEM (TS) or shared memory (SS), N in {32,64,128,256},
// with W issuer warps (one elected lane each) writing their own accumulators.
// One CTA per SM (dynamic shared memory > half the SM).  Every wait bounded.
#include <cstdio>
#include <cstdint>
#include <vector>
#include <algorithm>
#include <cuda_runtime.h>

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}
__host__ __device__ constexpr uint32_t idesc(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__global__ void __launch_bounds__(256, 1) rate(int mode, int N, int W, int iters, long long* cyc, int* err) {
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ uint32_t tslot;
  __shared__ __align__(8) uint64_t done[8];
  const uint32_t pad = (1024u - (su32(sm) & 1023u)) & 1023u;
  unsigned char* bsm = sm + pad;         // B: 256 rows x 128 B = 32 KB, 1 KB aligned
  unsigned char* asm_ = bsm + 32768;     // A (SS): 128 rows x 128 B = 16 KB
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < (32768 + 16384 + 1024) / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x3c003c00u;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&done[i])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&tslot)) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tbase = tslot;
  // A in TMEM at columns 256..319 (4 K-steps x 8 columns; contents zero after alloc are undefined -> write)
  if (warp < 4) {
    const uint32_t taddr = tbase + (static_cast<uint32_t>(warp * 32) << 16) + 256;
    for (int c = 0; c < 64; c += 8)
      asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1};" ::"r"(taddr + c),
                   "r"(0x3c003c00u)
                   : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp < W && lane == 0) {
    const uint32_t id = idesc(128, N);
    const uint32_t d = tbase + static_cast<uint32_t>(warp * N);  // W * N <= 256
    long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      const int k = i & 3;
      const uint64_t bd = sdesc(su32(bsm) + k * 32);
      const uint32_t acc = i > 0 ? 1u : 0u;
      if (mode == 0) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
            "r"(tbase + 256u + k * 8u), "l"(bd), "r"(id), "r"(acc)
            : "memory");
      } else {
        const uint64_t ad = sdesc(su32(asm_) + k * 32);
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(ad), "l"(bd), "r"(id), "r"(acc)
            : "memory");
      }
    }
    long long t1 = clock64();
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(&done[warp]))
                 : "memory");
    bool ok = false;
    for (uint32_t i = 0; i < (1u << 24) && !ok; ++i) {
      uint32_t r;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(r) : "r"(su32(&done[warp])) : "memory");
      ok = r != 0;
    }
    long long t2 = clock64();
    if (!ok) atomicOr(err, 1);
    cyc[(blockIdx.x * 8 + warp) * 2 + 0] = t1 - t0;
    cyc[(blockIdx.x * 8 + warp) * 2 + 1] = t2 - t0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tbase) : "memory");
}

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const int smem = 130 * 1024;
  cudaFuncSetAttribute(rate, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  long long* cyc;
  int* err;
  cudaMalloc(&cyc, sms * 16 * sizeof(long long));
  cudaMalloc(&err, 4);
  cudaMemset(err, 0, 4);
  const int iters = 4096;
  printf("SMs %d, %d MMAs per issuer\n", sms, iters);
  for (int mode = 0; mode < 2; ++mode)
    for (int N : {32, 64, 128, 256})
      for (int W : {1, 2, 3, 4, 6, 8}) {
        if (W * N > 256) continue;
        for (int rep = 0; rep < 2; ++rep) rate<<<sms, 256, smem>>>(mode, N, W, iters, cyc, err);
        cudaError_t e = cudaDeviceSynchronize();
        std::vector<long long> h(sms * 16);
        cudaMemcpy(h.data(), cyc, h.size() * sizeof(long long), cudaMemcpyDeviceToHost);
        std::vector<double> tot;
        for (int b = 0; b < sms; ++b) {
          long long mx = 0;
          for (int w = 0; w < W; ++w) mx = std::max(mx, h[(b * 8 + w) * 2 + 1]);
          tot.push_back(static_cast<double>(mx));
        }
        std::sort(tot.begin(), tot.end());
        const double med = tot[tot.size() / 2];
        const double per = med / (static_cast<double>(iters) * W);
        const double ideal = 128.0 * N * 16 * 2 / 8192.0;
        printf("%s N=%3d W=%d: %7.1f cycles per MMA across the SM (ideal %5.1f, %.2f of peak) %s\n",
               mode == 0 ? "TS" : "SS", N, W, per, ideal, ideal / per, cudaGetErrorString(e));
      }
  int herr = 0;
  cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  printf("err %d\n", herr);
  return 0;
}
