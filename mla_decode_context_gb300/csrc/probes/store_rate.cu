// Probe: how fast one SM writes a decode unit's partial output (128 rows x
// 512 fp32 = 256 KB) to global memory, in the epilogue's pattern, by
//   0: st.global of 16 bytes per lane from registers, four 128-byte row
//      pieces per warp instruction (the decode's current epilogue), or
//   1: bulk asynchronous stores (cp.async.bulk.global.shared::cta) of whole
//      512-byte row pieces out of shared memory, one per lane.
// Eight warps per CTA as in the decode's value CTA; each CTA writes its own
// 256 KB region `reps` times.  Run on every SM and on a quarter of them.
#include <cstdio>
#include <cstdint>
#include <vector>
#include <cuda_runtime.h>

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

constexpr int kRows = 128, kCols = 512, kWarps = 8;

__global__ void __launch_bounds__(32 * kWarps, 1) store_rate(int mode, int reps, float* out, int* err) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q4 = warp & 3, half = warp >> 2;
  float* base = out + static_cast<size_t>(blockIdx.x) * kRows * kCols;
  // mode 1: this warp's 32 rows x 128 columns (a quarter of its half rows) at
  // a time, 512 bytes per row piece, 16 KB per warp
  float* scr = reinterpret_cast<float*>(sm) + warp * (32 * 128);
  for (int i = threadIdx.x; i < kWarps * 32 * 128; i += blockDim.x) reinterpret_cast<float*>(sm)[i] = 1.0f;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  for (int rep = 0; rep < reps; ++rep) {
    if (mode == 0) {
      for (int c = half * 8; c < half * 8 + 8; ++c) {
        float* orow0 = base + (q4 * 32) * kCols;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int rr = 4 * m + (lane >> 3);
          *reinterpret_cast<float4*>(orow0 + rr * kCols + 32 * c + 4 * (lane & 7)) =
              make_float4(1.f, 2.f, 3.f, static_cast<float>(rep));
        }
      }
    } else {
      for (int part = 0; part < 2; ++part) {
        const int row = q4 * 32 + lane;
        float* dst = base + row * kCols + half * 256 + part * 128;
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                     "r"(su32(scr + lane * 128)), "r"(512u)
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      }
    }
  }
  if (mode == 1) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  if (threadIdx.x == 0 && base[0] == -1.f) atomicOr(err, 1);
}

static float run(int mode, int ctas, int reps, float* out, int* err) {
  const int smem = kWarps * 32 * 128 * 4;  // 128 KB
  cudaFuncSetAttribute(store_rate, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  float best = 1e30f;
  for (int r = 0; r < 4; ++r) {
    cudaEventRecord(e0);
    store_rate<<<ctas, 32 * kWarps, smem>>>(mode, reps, out, err);
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms;
    cudaEventElapsedTime(&ms, e0, e1);
    if (r > 0 && ms < best) best = ms;
  }
  return best;
}

int main() {
  int sms = 0, clk = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, 0);
  float* out = nullptr;
  int* err = nullptr;
  const size_t bytes = static_cast<size_t>(sms) * kRows * kCols * 4;
  if (cudaMalloc(&out, bytes) != cudaSuccess || cudaMalloc(&err, 4) != cudaSuccess) {
    printf("alloc failed\n");
    return 1;
  }
  cudaMemset(out, 0, bytes);
  cudaMemset(err, 0, 4);
  const int reps = 50;
  printf("SMs %d, clock %d kHz, 256 KB per CTA x %d reps\n", sms, clk, reps);
  const char* names[2] = {"st.global 16 B per lane", "bulk stores, 512 B per row piece"};
  for (int ctas : {sms, sms / 4})
    for (int mode = 0; mode < 2; ++mode) {
      const float ms = run(mode, ctas, reps, out, err);
      const double moved = static_cast<double>(ctas) * reps * kRows * kCols * 4;
      printf("%3d CTAs, %-34s %8.3f ms  %8.1f GB/s  %5.1f B/clk/SM  (%.0f cycles per 256 KB)\n", ctas, names[mode], ms,
             moved / (ms * 1e6), moved / (ms * 1e-3) / ctas / (clk * 1e3),
             (ms * 1e-3) * (clk * 1e3) / reps);
    }
  int h = 0;
  cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost);
  printf("err %d, cuda %s\n", h, cudaGetErrorString(cudaGetLastError()));
  return 0;
}
