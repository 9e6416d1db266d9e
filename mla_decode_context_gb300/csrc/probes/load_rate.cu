// Probe: per-SM global->shared streaming rate of 16-byte cp.async vs
// LDG.128 + STS.128, in the decode producers' pattern (rows of 640 bytes out
// of 1152-byte cache rows, 8 lanes per 128-byte line, stages of 32 rows x 5
// chunks).  One CTA per SM; a consumer warp frees each stage as soon as it has
// landed.  Every wait is bounded.  Run on every SM (HBM-bound) and on a
// quarter of them (the SM's own ceiling).
#include <cstdio>
#include <cstdint>
#include <vector>
#include <cuda_runtime.h>

constexpr int kStages = 5, kRows = 32, kNch = 5, kChunk = kRows * 128, kStageBytes = kNch * kChunk;
constexpr int kRowBytes = 1152;

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void minit(uint64_t* b, uint32_t c) { asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(c) : "memory"); }
__device__ __forceinline__ void marrive(uint64_t* b) { asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory"); }
__device__ __forceinline__ bool mtest(uint64_t* b, uint32_t par) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(ok) : "r"(su32(b)), "r"(par) : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mwait(uint64_t* b, uint32_t par) {
  for (uint32_t i = 0; i < (1u << 22); ++i) if (mtest(b, par)) return true;
  return false;
}

template <int kMode, int kProdWarps>  // 0: cp.async, 1: ldg+sts
__global__ void __launch_bounds__(32 * (kProdWarps + 1), 1) probe(const unsigned char* __restrict__ kv, int64_t nrows_total, int tiles, int* err) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ uint64_t full[kStages], freeb[kStages];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kGroupWarps = kProdWarps / 2, kGroupThreads = 32 * kGroupWarps;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) { minit(&full[i], kGroupThreads); minit(&freeb[i], 1); }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // this CTA's rows: a contiguous range far from the others (no L2 reuse)
  const int64_t base_row = static_cast<int64_t>(blockIdx.x) * tiles * kRows;
  if (warp < kProdWarps) {
    const int group = warp / kGroupWarps, gw = warp % kGroupWarps;
    const int x = lane & 7;
    constexpr int kRowsPerWarp = kRows / kGroupWarps;  // 8 (4 warps) or 4 (8 warps)
    bool ok = true;
    for (int j = group; j < tiles && ok; j += 2) {
      const int st = j % kStages;
      ok = mwait(&freeb[st], ((j / kStages) & 1) ^ 1);
      if (!ok) break;
      const uint32_t sb = su32(smem) + st * kStageBytes;
      for (int rr = lane >> 3; rr < kRowsPerWarp; rr += 4) {
        const int row = gw * kRowsPerWarp + rr;
        const int64_t grow = base_row + static_cast<int64_t>(j) * kRows + row;
        const unsigned char* src = kv + grow * kRowBytes + x * 16;
        const uint32_t swz = row * 128 + ((x ^ (row & 7)) << 4);
#pragma unroll
        for (int c = 0; c < kNch; ++c) {
          if (kMode == 0) {
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sb + c * kChunk + swz), "l"(src + c * 128) : "memory");
          } else {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + c * 128));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sb + c * kChunk + swz), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
          }
        }
      }
      if (kMode == 0) asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(su32(&full[st])) : "memory");
      else marrive(&full[st]);
    }
    if (!ok) atomicOr(err, 1);
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // consumer: free each stage once it has landed
    bool ok = true;
    for (int j = 0; j < tiles && ok; ++j) {
      const int st = j % kStages;
      ok = mwait(&full[st], (j / kStages) & 1);
      if (ok && lane == 0) marrive(&freeb[st]);
      __syncwarp();
    }
    if (!ok) atomicOr(err, 2);
  }
}

template <int M, int W>
float run(const unsigned char* kv, int64_t nrows, int ctas, int tiles, int* err) {
  const size_t smem = 120 * 1024;  // one CTA per SM
  cudaFuncSetAttribute(probe<M, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0); cudaEventCreate(&e1);
  float best = 1e30f;
  for (int rep = 0; rep < 5; ++rep) {
    cudaEventRecord(e0);
    probe<M, W><<<ctas, 32 * (W + 1), smem>>>(kv, nrows, tiles, err);
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms; cudaEventElapsedTime(&ms, e0, e1);
    if (rep > 0 && ms < best) best = ms;
  }
  return best;
}

int main() {
  int dev = 0, sms = 0, clk = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev);
  const int tiles = 400;  // per CTA: 400 x 32 rows x 640 B = 8.2 MB
  const int ctas = sms;
  const int64_t nrows = static_cast<int64_t>(ctas) * tiles * kRows;   // every row read once
  const size_t bytes = static_cast<size_t>(nrows) * kRowBytes;        // ~2.2 GB of cache rows
  unsigned char* kv = nullptr;
  int* err = nullptr;
  if (cudaMalloc(&kv, bytes) != cudaSuccess || cudaMalloc(&err, 4) != cudaSuccess) { printf("alloc failed\n"); return 1; }
  cudaMemset(kv, 1, bytes);
  cudaMemset(err, 0, 4);
  const double moved = static_cast<double>(nrows) * kNch * 128;  // bytes delivered to shared memory
  struct R { const char* name; float ms; };
  std::vector<R> rs;
  rs.push_back({"cp.async, 8 producer warps", run<0, 8>(kv, nrows, ctas, tiles, err)});
  rs.push_back({"cp.async, 16 producer warps", run<0, 16>(kv, nrows, ctas, tiles, err)});
  rs.push_back({"ldg+sts, 8 producer warps", run<1, 8>(kv, nrows, ctas, tiles, err)});
  rs.push_back({"ldg+sts, 16 producer warps", run<1, 16>(kv, nrows, ctas, tiles, err)});
  // A quarter of the SMs: HBM no longer bounds the stream, so the rate per
  // SM is the SM's own ceiling.
  const int q = sms / 4;
  const double moved_q = static_cast<double>(q) * tiles * kRows * kNch * 128;
  const float q8 = run<0, 8>(kv, nrows, q, tiles, err);
  const float q16 = run<0, 16>(kv, nrows, q, tiles, err);
  int h_err = 0;
  cudaMemcpy(&h_err, err, 4, cudaMemcpyDeviceToHost);
  printf("SMs %d, clock %d kHz, %d CTAs x %d tiles, %.1f MB moved, err %d, cuda %s\n", sms, clk, ctas, tiles, moved / 1e6, h_err,
         cudaGetErrorString(cudaGetLastError()));
  for (auto& r : rs)
    printf("%-30s %8.3f ms  %7.1f GB/s  %5.1f B/clk/SM (at the %.2f GHz maximum clock)\n", r.name, r.ms,
           moved / (r.ms * 1e6), moved / (r.ms * 1e-3) / ctas / (clk * 1e3), clk * 1e-6);
  printf("%d CTAs only:\n", q);
  printf("%-30s %8.3f ms  %7.1f GB/s  %5.1f B/clk/SM\n", "cp.async, 8 producer warps", q8, moved_q / (q8 * 1e6),
         moved_q / (q8 * 1e-3) / q / (clk * 1e3));
  printf("%-30s %8.3f ms  %7.1f GB/s  %5.1f B/clk/SM\n", "cp.async, 16 producer warps", q16, moved_q / (q16 * 1e6),
         moved_q / (q16 * 1e-3) / q / (clk * 1e3));
  cudaFree(kv); cudaFree(err);
  return 0;
}
