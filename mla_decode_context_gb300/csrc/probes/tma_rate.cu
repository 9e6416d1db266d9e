// Probe: TMA streaming of shard-strided KV boxes (120k geometry: 64-row
// blocks, D=8 shards, interleave 1 -> each (block, shard) box = 8 rows x 9
// chunks = 9 KB), vs ring depth, with and without cluster pairing/multicast.
// Every wait is bounded; the bounds of every box are checked on the host.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include <vector>
#include <algorithm>
#include <random>

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s at %d: %s\n", #x, __LINE__, cudaGetErrorString(e_)); exit(1); } } while (0)

constexpr int kNB = 3750;        // blocks (276 MB: above L2)
constexpr int kBS = 64, kD = 8, kRow = 1152;
constexpr int kBoxBytes = 9 * 8 * 128;  // 9216
constexpr uint32_t kLimit = 1u << 22;

__device__ int g_err;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) { asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory"); }
__device__ __forceinline__ void expect_tx(uint64_t* b, uint32_t n) { asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory"); }
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t par) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(ok) : "r"(su32(b)), "r"(par) : "memory");
  return ok;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t par) {
  for (uint32_t i = 0; i < kLimit; ++i) if (mbar_test(b, par)) return true;
  return false;
}
__device__ __forceinline__ void tma5(const CUtensorMap* m, void* dst, uint64_t* bar, int c4) {
  asm volatile("cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %3, %3, %3, %2}], [%4];"
               ::"r"(su32(dst)), "l"(m), "r"(c4), "r"(0), "r"(su32(bar)) : "memory");
}
__device__ __forceinline__ void tma5_mc(const CUtensorMap* m, void* dst, uint64_t* bar, int c4, uint16_t mask) {
  asm volatile("cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1, {%3, %3, %3, %3, %2}], [%4], %5;"
               ::"r"(su32(dst)), "l"(m), "r"(c4), "r"(0), "r"(su32(bar)), "h"(mask) : "memory");
}
__device__ __forceinline__ uint32_t ctarank() { uint32_t r; asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r)); return r; }
__device__ __forceinline__ void cluster_sync() { asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t mapa(uint32_t a, uint32_t r) { uint32_t o; asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(o) : "r"(a), "r"(r)); return o; }
__device__ __forceinline__ void arrive_remote(uint32_t a) { asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(a) : "memory"); }

// mode 0: each CTA streams its own boxes.  mode 1: 2-CTA clusters, both CTAs
// load the same boxes.  mode 2: 2-CTA clusters, each box multicast once to
// both (slot s issued by rank s % 2, refilled once both CTAs consumed it).
template <int kMode>
__global__ void probe(const __grid_constant__ CUtensorMap m, const int* __restrict__ perm, int nbox, int nunits, int ns) {
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* ring = (unsigned char*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[32], consumed[32];
  const int unit = kMode == 0 ? blockIdx.x : blockIdx.x / 2;
  const uint32_t rank = kMode == 0 ? 0 : ctarank();
  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) { mbar_init(&full[s], 1); mbar_init(&consumed[s], 2); }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (kMode != 0) cluster_sync();
  if (threadIdx.x == 0) {
    // like a split of one shard: unit u walks blocks [(u / D) * per_unit, ...) of shard u % D
    const int groups = (nunits + kD - 1) / kD;
    const int per_unit = (kNB + groups - 1) / groups;
    const int blk0 = (unit / kD) * per_unit, shard = unit % kD;
    auto row0 = [&](int i) { return perm[blk0 + i] * kBS + shard; };
    int issued = 0, done = 0;
    const int mine = max(0, min(per_unit, kNB - blk0));
    // prologue
    for (int s = 0; s < ns && issued < mine; ++s, ++issued) {
      expect_tx(&full[s], kBoxBytes);
      const int b = issued;
      if (kMode == 2) { if ((s & 1) == (int)rank) tma5_mc(&m, ring + s * kBoxBytes, &full[s], row0(b), 0x3); }
      else tma5(&m, ring + s * kBoxBytes, &full[s], row0(b));
    }
    bool ok = true;
    while (done < mine && ok) {
      const int s = done % ns;
      const uint32_t par = (done / ns) & 1;
      ok = mbar_wait(&full[s], par);
      if (!ok) break;
      ++done;
      const int sl = issued % ns;  // == s while refills remain
      if (kMode == 2) {
        // re-arm first, then tell the slot's issuer that this CTA consumed it
        if (issued < mine) expect_tx(&full[sl], kBoxBytes);
        arrive_remote(mapa(su32(&consumed[s]), s & 1));
      }
      if (issued < mine) {
        const int b = issued;
        if (kMode == 2) {
          if ((sl & 1) == (int)rank) {
            ok = mbar_wait(&consumed[sl], ((issued / ns) - 1) & 1);
            if (!ok) break;
            tma5_mc(&m, ring + sl * kBoxBytes, &full[sl], row0(b), 0x3);
          }
        } else {
          expect_tx(&full[sl], kBoxBytes);
          tma5(&m, ring + sl * kBoxBytes, &full[sl], row0(b));
        }
        ++issued;
      }
    }
    if (!ok) atomicExch(&g_err, 1 + (int)blockIdx.x);
    // drain: wait for every issued copy into this CTA (bounded)
    for (; done < issued; ++done) mbar_wait(&full[done % ns], (done / ns) & 1);
  }
  __syncthreads();
  if (kMode != 0) cluster_sync();
}

// mode 3: like mode 0 with `nw` issuing warps per CTA, each streaming its
// own share of the CTA's boxes through its own part of the ring (ns slots
// per warp).  box_bytes / rows_per_box describe the map (strided 8-row boxes
// or contiguous 32-row boxes).
__global__ void probe_mw(const __grid_constant__ CUtensorMap m, const int* __restrict__ perm, int nunits, int ns, int nw,
                         int box_bytes, int boxes_per_block, int rows_step) {
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* ring = (unsigned char*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[64];
  const int w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < ns * nw; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0 && w < nw) {
    const int unit = blockIdx.x;
    // strided boxes: unit u walks shard u % D of its block group; contiguous
    // boxes: every unit its own blocks
    const int groups = boxes_per_block == 1 ? (nunits + kD - 1) / kD : nunits;
    const int per_unit = (kNB + groups - 1) / groups;
    const int blk0 = (boxes_per_block == 1 ? unit / kD : unit) * per_unit, shard = unit % kD;
    const int nblk = max(0, min(per_unit, kNB - blk0));
    const int total = nblk * boxes_per_block;      // boxes of this unit
    // warp w takes boxes w, w + nw, ...
    const int mine = total > w ? (total - w + nw - 1) / nw : 0;
    auto coord = [&](int k) {
      const int b = w + k * nw;
      const int blk = blk0 + b / boxes_per_block, sub = b % boxes_per_block;
      return boxes_per_block == 1 ? perm[blk] * kBS + shard : perm[blk] * kBS + sub * rows_step;
    };
    uint64_t* f = full + w * ns;
    unsigned char* rg = ring + (size_t)w * ns * box_bytes;
    int issued = 0, done = 0;
    for (; issued < ns && issued < mine; ++issued) { expect_tx(&f[issued], box_bytes); tma5(&m, rg + issued * box_bytes, &f[issued], coord(issued)); }
    bool ok = true;
    while (done < mine && ok) {
      const int s = done % ns;
      ok = mbar_wait(&f[s], (done / ns) & 1);
      if (!ok) break;
      ++done;
      if (issued < mine) { const int sl = issued % ns; expect_tx(&f[sl], box_bytes); tma5(&m, rg + sl * box_bytes, &f[sl], coord(issued)); ++issued; }
    }
    if (!ok) atomicExch(&g_err, 1 + (int)blockIdx.x);
    for (; done < issued; ++done) mbar_wait(&f[done % ns], (done / ns) & 1);
  }
  __syncthreads();
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                             const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                             CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int main() {
  int sms = 0; CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  void* fn = nullptr; cudaDriverEntryPointQueryResult q;
  CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
  if (!fn || q != cudaDriverEntryPointSuccess) { printf("no encode fn\n"); return 1; }
  EncodeFn enc = (EncodeFn)fn;
  const size_t cache_bytes = (size_t)kNB * kBS * kRow;
  void* kv; CK(cudaMalloc(&kv, cache_bytes)); CK(cudaMemset(kv, 0, cache_bytes));
  void* flush; CK(cudaMalloc(&flush, 512u << 20));
  std::vector<int> perm(kNB); for (int i = 0; i < kNB; ++i) perm[i] = i;
  std::shuffle(perm.begin(), perm.end(), std::mt19937(1));
  int* dperm; CK(cudaMalloc(&dperm, kNB * 4)); CK(cudaMemcpy(dperm, perm.data(), kNB * 4, cudaMemcpyHostToDevice));
  // 5-D view: (e 64 | i 1 [1152] | per 8 [9216] | c 9 [128] | row0 nb*64 [1152])
  CUtensorMap m;
  cuuint64_t dims[5] = {64, 1, (cuuint64_t)(kBS / kD), 9, (cuuint64_t)kNB * kBS};
  cuuint64_t strides[4] = {kRow, (cuuint64_t)kD * kRow, 128, kRow};
  cuuint32_t box[5] = {64, 1, (cuuint32_t)(kBS / kD), 9, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, kv, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  printf("encode 5d shard-strided map: %d\n", (int)r);
  if (r != CUDA_SUCCESS) return 1;
  const int nbox = kNB * kD;
  // host bounds check of every box: rows row0 + 8*per, per < 8, inside the cache
  for (int b = 0; b < nbox; ++b) {
    long row0 = (long)perm[b / kD] * kBS + b % kD;
    long last = row0 + (kBS / kD - 1) * kD;
    if (row0 < 0 || last >= (long)kNB * kBS) { printf("box %d out of bounds\n", b); return 1; }
  }
  cudaEvent_t e0, e1; CK(cudaEventCreate(&e0)); CK(cudaEventCreate(&e1));
  int zero = 0;
  for (int mode = 0; mode < 3; ++mode) {
    for (int ns : {4, 8, 12, 16, 20}) {
      const size_t smem = (size_t)ns * kBoxBytes + 1024;
      int units = mode == 0 ? sms : sms / 2;
      float best = 1e9;
      for (int rep = 0; rep < 3; ++rep) {
        CK(cudaMemcpyToSymbol(g_err, &zero, 4));
        CK(cudaMemsetAsync(flush, rep, 512u << 20));
        CK(cudaEventRecord(e0));
        if (mode == 0) {
          CK(cudaFuncSetAttribute(probe<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
          probe<0><<<units, 32, smem>>>(m, dperm, nbox, units, ns);
        } else {
          cudaLaunchConfig_t cfg = {}; cudaLaunchAttribute at[1];
          cfg.gridDim = dim3(2 * units); cfg.blockDim = dim3(32); cfg.dynamicSmemBytes = smem;
          at[0].id = cudaLaunchAttributeClusterDimension; at[0].val.clusterDim.x = 2; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
          cfg.attrs = at; cfg.numAttrs = 1;
          if (mode == 1) { CK(cudaFuncSetAttribute(probe<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)); CK(cudaLaunchKernelEx(&cfg, probe<1>, m, (const int*)dperm, nbox, units, ns)); }
          else { CK(cudaFuncSetAttribute(probe<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)); CK(cudaLaunchKernelEx(&cfg, probe<2>, m, (const int*)dperm, nbox, units, ns)); }
        }
        CK(cudaEventRecord(e1));
        CK(cudaEventSynchronize(e1));
        CK(cudaGetLastError());
        float ms; CK(cudaEventElapsedTime(&ms, e0, e1));
        int err = 0; CK(cudaMemcpyFromSymbol(&err, g_err, 4));
        if (err) { printf("mode %d ns %d: wait timed out (block %d)\n", mode, ns, err - 1); return 1; }
        best = std::min(best, ms);
      }
      long boxes = 0;
      { const int groups = (units + kD - 1) / kD, per_unit = (kNB + groups - 1) / groups;
        for (int u = 0; u < units; ++u) boxes += std::max(0, std::min(per_unit, kNB - (u / kD) * per_unit)); }
      printf("mode %d (%s) ring %2d x 9 KB: %.3f ms  %.0f GB/s of unique bytes (%ld boxes)\n", mode,
             mode == 0 ? "1 CTA/SM own boxes" : mode == 1 ? "pairs, both load" : "pairs, multicast", ns, best,
             (double)boxes * kBoxBytes / (best * 1e-3) / 1e9, boxes);
    }
  }
  // contiguous-rows map: (e 64 | rows 32 [1152] | c 9 [128] | - 1 | row0 [1152]) box 32 rows x 9 chunks = 36 KB
  CUtensorMap mc;
  {
    cuuint64_t d2[5] = {64, 32, 9, 1, (cuuint64_t)kNB * kBS};
    cuuint64_t s2[4] = {kRow, 128, 128, kRow};
    cuuint32_t b2[5] = {64, 32, 9, 1, 1};
    CUresult r2 = enc(&mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, kv, d2, s2, b2, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    printf("encode contiguous map: %d\n", (int)r2);
    if (r2 != CUDA_SUCCESS) return 1;
    // every box: rows perm*64 + {0, 32} .. +31 inside the cache
    for (int b = 0; b < kNB; ++b) if ((long)perm[b] * kBS + 32 + 31 >= (long)kNB * kBS) { printf("oob\n"); return 1; }
  }
  struct Cfg { const CUtensorMap* m; const char* name; int box; int bpb; int step; int ns; int nw; int ctas_per_sm; };
  std::vector<Cfg> cfgs = {
    {&m, "strided 9 KB, 1 warp", kBoxBytes, 1, 0, 16, 1, 1},
    {&m, "strided 9 KB, 2 warps", kBoxBytes, 1, 0, 8, 2, 1},
    {&m, "strided 9 KB, 4 warps", kBoxBytes, 1, 0, 4, 4, 1},
    {&m, "strided 9 KB, 1 warp, 2 CTA/SM", kBoxBytes, 1, 0, 8, 1, 2},
    {&mc, "contig 36 KB, 1 warp", 36864, 2, 32, 5, 1, 1},
    {&mc, "contig 36 KB, 2 warps", 36864, 2, 32, 2, 2, 1},
  };
  for (auto& c : cfgs) {
    const size_t smem = (size_t)c.ns * c.nw * c.box + 1024;
    CK(cudaFuncSetAttribute(probe_mw, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    const int units = sms * c.ctas_per_sm;
    float best = 1e9;
    for (int rep = 0; rep < 3; ++rep) {
      CK(cudaMemcpyToSymbol(g_err, &zero, 4));
      CK(cudaMemsetAsync(flush, rep, 512u << 20));
      CK(cudaEventRecord(e0));
      probe_mw<<<units, 32 * c.nw, smem>>>(*c.m, dperm, units, c.ns, c.nw, c.box, c.bpb, c.step);
      CK(cudaEventRecord(e1));
      CK(cudaEventSynchronize(e1));
      CK(cudaGetLastError());
      float ms; CK(cudaEventElapsedTime(&ms, e0, e1));
      int err = 0; CK(cudaMemcpyFromSymbol(&err, g_err, 4));
      if (err) { printf("%s: wait timed out\n", c.name); return 1; }
      best = std::min(best, ms);
    }
    long bytes = 0;
    { const int groups = c.bpb == 1 ? (units + kD - 1) / kD : units, per_unit = (kNB + groups - 1) / groups;
      for (int u = 0; u < units; ++u)
        bytes += (long)std::max(0, std::min(per_unit, kNB - (c.bpb == 1 ? u / kD : u) * per_unit)) * c.bpb * c.box; }
    printf("%-36s: %.3f ms  %.0f GB/s\n", c.name, best, bytes / (best * 1e-3) / 1e9);
  }
  return 0;
}
