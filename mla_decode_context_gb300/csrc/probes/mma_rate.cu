// Probe: tcgen05.mma kind::f16 issue/execution rate, M=128, K=16, bf16, fp32
// accumulators, A from TMEM (TS) or shared memory (SS), N in {32,64,128,256},
// with W issuer warps (one elected lane each) writing their own accumulators.
// A second sweep has each issuing lane drive A accumulators round-robin, which
// tells whether the ~121-cycle step of one issuer is the issuing thread's or
// the accumulator chain's.  A third sweep has L lanes of each issuing warp
// execute the same tcgen05.mma (each lane its own accumulator) from a loop
// with no arithmetic between the MMAs.  A fourth runs six such issuers next
// to K warps of one kind of other work (mbarrier polls, blocking mbarrier
// waits, cp.async streams from HBM, TMEM loads, shared-memory loads) to see
// which of them slows the issue.
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

__global__ void __launch_bounds__(256, 1) rate(int mode, int N, int W, int A, int iters, long long* cyc, int* err) {
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
    const uint32_t d0 = tbase + static_cast<uint32_t>(warp * A * N);  // W * A * N <= 256
    long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      const int a = i % A;
      const int k = (i / A) & 3;
      const uint32_t d = d0 + static_cast<uint32_t>(a * N);
      const uint64_t bd = sdesc(su32(bsm) + k * 32);
      const uint32_t acc = i >= A ? 1u : 0u;
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

// W warps x L lanes, every lane its own N=32 accumulator (W * L <= 8), the
// loop unrolled over the four k-steps so that nothing but the MMA is issued.
__global__ void __launch_bounds__(256, 1) rate_lanes(int W, int L, int iters, long long* cyc, int* err) {
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ uint32_t tslot;
  __shared__ __align__(8) uint64_t done[8];
  const uint32_t pad = (1024u - (su32(sm) & 1023u)) & 1023u;
  unsigned char* bsm = sm + pad;
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
  if (warp < W && lane < L) {
    const int q = warp * L + lane;  // < 8
    const uint32_t id = idesc(128, 32);
    const uint32_t d = tbase + static_cast<uint32_t>(q * 32);
    const uint32_t a0 = tbase + 256u;
    const uint64_t bd0 = sdesc(su32(bsm));
    long long t0 = clock64();
    for (int i = 0; i < iters; i += 4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t acc = (i + k) > 0 ? 1u : 0u;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
            "r"(a0 + k * 8u), "l"(bd0 + 2u * k), "r"(id), "r"(acc)
            : "memory");
      }
    }
    long long t1 = clock64();
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(&done[q]))
                 : "memory");
    bool ok = false;
    for (uint32_t i = 0; i < (1u << 24) && !ok; ++i) {
      uint32_t r;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(r) : "r"(su32(&done[q])) : "memory");
      ok = r != 0;
    }
    long long t2 = clock64();
    if (!ok) atomicOr(err, 1);
    cyc[(blockIdx.x * 8 + q) * 2 + 0] = t1 - t0;
    cyc[(blockIdx.x * 8 + q) * 2 + 1] = t2 - t0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tbase) : "memory");
}

// Six unrolled issuers (warps 0-5, N = 32, own accumulators) next to K noise
// warps (warps 8 .. 8 + K - 1) doing kind `noise` until the issuers are done.
__global__ void __launch_bounds__(768, 1) rate_noise(int noise, int K, int W, int spread, int iters, const uint4* gbuf,
                                                     size_t gwords,
                                                     long long* cyc, int* err) {
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ uint32_t tslot;
  __shared__ __align__(8) uint64_t done[8];
  __shared__ __align__(8) uint64_t never;
  __shared__ volatile int finished;
  const uint32_t pad = (1024u - (su32(sm) & 1023u)) & 1023u;
  unsigned char* bsm = sm + pad;               // B operand: 32 KB
  unsigned char* scratch = bsm + 49152;        // noise: 16 warps x 4 KB
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 36864 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(bsm)[i] = 0x3c003c00u;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&done[i])) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&never)) : "memory");
    finished = 0;
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
  if (warp < 6) {
    if (lane == 0 && warp < W) {
      const uint32_t id = idesc(128, 32);
      const uint32_t d = tbase + static_cast<uint32_t>(warp * 32);
      const uint32_t a0 = tbase + 256u;
      const uint64_t bd0 = sdesc(su32(bsm));
      uint64_t bc = bd0;  // spread: the chunk of this group of four k-steps (nine 4 KB chunks, as a stage)
      int c = 0;
      long long t0 = clock64();
      for (int i = 0; i < iters; i += 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t acc = (i + k) > 0 ? 1u : 0u;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
              "r"(a0 + k * 8u), "l"(bc + 2u * k), "r"(id), "r"(acc)
              : "memory");
        }
        if (spread) {
          bc += 4096 >> 4;
          if (++c == 9) { c = 0; bc = bd0; }
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
      if (!ok) atomicOr(err, 1);
      cyc[(blockIdx.x * 8 + warp) * 2 + 0] = t1 - t0;
      atomicAdd(const_cast<int*>(&finished), 1);
    }
    __syncwarp();
  } else if (warp >= 8 && warp < 8 + K) {
    const uint32_t my = su32(scratch + (warp - 8) * 4096);
    const size_t span = gwords / gridDim.x;  // this CTA's share of the buffer, in 16-byte words
    const uint4* gsrc = gbuf + blockIdx.x * span;
    size_t g = static_cast<size_t>((warp - 8) * 512 + lane);
    uint32_t sink = 0;
    for (uint32_t it = 0; it < (1u << 22) && finished < W; ++it) {
      if (noise == 0) {  // non-blocking mbarrier polls
        uint32_t r;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(r) : "r"(su32(&never)) : "memory");
        sink += r;
      } else if (noise == 1) {  // blocking mbarrier waits (each returns after the hardware's time limit)
        uint32_t r;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(r) : "r"(su32(&never)) : "memory");
        sink += r;
      } else if (noise == 2) {  // cp.async stream: 4 x 16 B per lane per round, 8 rounds in flight
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t dst = my + static_cast<uint32_t>(((it & 7) * 4 + c) & 7) * 512 + lane * 16;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(gsrc + g) : "memory");
          g += 32;
          if (g >= span) g -= span;
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 8;" ::: "memory");
      } else if (noise == 3) {  // TMEM loads, 32 columns at a time
        const uint32_t taddr = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 320;
        uint32_t v[8];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                     : "r"(taddr + 8 * (it & 3))
                     : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        sink += v[0] ^ v[7];
      } else {  // shared-memory loads
        uint32_t v;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(my + ((it * 128 + lane * 4) & 4095)) : "memory");
        sink += v;
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (sink == 0x12345678u) atomicOr(err, 2);
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
        for (int rep = 0; rep < 2; ++rep) rate<<<sms, 256, smem>>>(mode, N, W, 1, iters, cyc, err);
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
  // One lane driving several accumulators, TS, N = 32.
  for (int W : {1, 2, 3, 4})
    for (int A : {1, 2, 3, 4}) {
      if (W * A * 32 > 256) continue;
      for (int rep = 0; rep < 2; ++rep) rate<<<sms, 256, smem>>>(0, 32, W, A, iters, cyc, err);
      cudaError_t e = cudaDeviceSynchronize();
      std::vector<long long> h(sms * 16);
      cudaMemcpy(h.data(), cyc, h.size() * sizeof(long long), cudaMemcpyDeviceToHost);
      std::vector<double> tot, issue;
      for (int b = 0; b < sms; ++b) {
        long long mx = 0, mi = 0;
        for (int w = 0; w < W; ++w) {
          mx = std::max(mx, h[(b * 8 + w) * 2 + 1]);
          mi = std::max(mi, h[(b * 8 + w) * 2 + 0]);
        }
        tot.push_back(static_cast<double>(mx));
        issue.push_back(static_cast<double>(mi));
      }
      std::sort(tot.begin(), tot.end());
      std::sort(issue.begin(), issue.end());
      const double per = tot[tot.size() / 2] / (static_cast<double>(iters) * W);
      const double per_lane = issue[issue.size() / 2] / static_cast<double>(iters);
      printf("TS N= 32 W=%d A=%d: %7.1f cycles per MMA across the SM, %7.1f cycles per issue of one lane %s\n", W, A,
             per, per_lane, cudaGetErrorString(e));
    }
  // L lanes of each of W warps issuing, unrolled loop, TS, N = 32.
  cudaFuncSetAttribute(rate_lanes, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  for (int W : {1, 2, 4, 8})
    for (int L : {1, 2, 4, 8}) {
      if (W * L > 8) continue;
      for (int rep = 0; rep < 2; ++rep) rate_lanes<<<sms, 256, smem>>>(W, L, iters, cyc, err);
      cudaError_t e = cudaDeviceSynchronize();
      std::vector<long long> h(sms * 16);
      cudaMemcpy(h.data(), cyc, h.size() * sizeof(long long), cudaMemcpyDeviceToHost);
      std::vector<double> tot, issue;
      for (int b = 0; b < sms; ++b) {
        long long mx = 0, mi = 0;
        for (int q = 0; q < W * L; ++q) {
          mx = std::max(mx, h[(b * 8 + q) * 2 + 1]);
          mi = std::max(mi, h[(b * 8 + q) * 2 + 0]);
        }
        tot.push_back(static_cast<double>(mx));
        issue.push_back(static_cast<double>(mi));
      }
      std::sort(tot.begin(), tot.end());
      std::sort(issue.begin(), issue.end());
      const double per = tot[tot.size() / 2] / (static_cast<double>(iters) * W * L);
      const double per_warp = issue[issue.size() / 2] / static_cast<double>(iters);
      printf("TS N= 32 unrolled W=%d L=%d: %7.1f cycles per MMA across the SM, %7.1f cycles per MMA instruction of one warp %s\n",
             W, L, per, per_warp, cudaGetErrorString(e));
    }
  // Six issuers next to K warps of other work.
  {
    const size_t gbytes = size_t(512) << 20;
    uint4* gbuf = nullptr;
    cudaMalloc(&gbuf, gbytes);
    cudaMemset(gbuf, 0, gbytes);
    const int smem2 = 49152 + 16 * 4096 + 1024;
    cudaFuncSetAttribute(rate_noise, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2);
    const char* kinds[5] = {"mbarrier test_wait polls", "mbarrier try_wait", "cp.async from HBM", "tcgen05.ld", "ld.shared"};
    for (int noise = 0; noise < 5; ++noise)
      for (int K : {0, 4, 8, 16}) {
        if (K == 0 && noise > 0) continue;
        for (int rep = 0; rep < 2; ++rep)
          rate_noise<<<sms, 768, smem2>>>(noise, K, 6, 0, iters, gbuf, gbytes / 16, cyc, err);
        cudaError_t e = cudaDeviceSynchronize();
        std::vector<long long> h(sms * 16);
        cudaMemcpy(h.data(), cyc, h.size() * sizeof(long long), cudaMemcpyDeviceToHost);
        std::vector<double> issue;
        for (int b = 0; b < sms; ++b) {
          long long mi = 0;
          for (int q = 0; q < 6; ++q) mi = std::max(mi, h[(b * 8 + q) * 2 + 0]);
          issue.push_back(static_cast<double>(mi));
        }
        std::sort(issue.begin(), issue.end());
        printf("6 issuers + %2d warps of %-26s: %7.1f cycles per MMA of one issuer (%.1f across the SM) %s\n", K,
               K ? kinds[noise] : "nothing", issue[issue.size() / 2] / iters, issue[issue.size() / 2] / iters / 6,
               cudaGetErrorString(e));
      }
    // B read from nine distinct 4 KB chunks (36 KB, as the decode's stage)
    // rather than one: W issuers, with or without cp.async streams
    for (int W : {3, 6})
      for (int spread : {0, 1})
        for (int K : {0, 8, 16}) {
          for (int rep = 0; rep < 2; ++rep)
            rate_noise<<<sms, 768, smem2>>>(2, K, W, spread, iters, gbuf, gbytes / 16, cyc, err);
          cudaError_t e = cudaDeviceSynchronize();
          std::vector<long long> h(sms * 16);
          cudaMemcpy(h.data(), cyc, h.size() * sizeof(long long), cudaMemcpyDeviceToHost);
          std::vector<double> issue;
          for (int b = 0; b < sms; ++b) {
            long long mi = 0;
            for (int q = 0; q < W; ++q) mi = std::max(mi, h[(b * 8 + q) * 2 + 0]);
            issue.push_back(static_cast<double>(mi));
          }
          std::sort(issue.begin(), issue.end());
          printf("%d issuers, B from %s, %2d cp.async warps: %7.1f cycles per MMA of one issuer %s\n", W,
                 spread ? "9 chunks" : "1 chunk ", K, issue[issue.size() / 2] / iters, cudaGetErrorString(e));
        }
    cudaFree(gbuf);
  }
  int herr = 0;
  cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  printf("err %d\n", herr);
  return 0;
}
