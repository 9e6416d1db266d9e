// Tensor-core split-KV MLA decode for sm_103a (tcgen05 + TMEM + TMA + DSMEM).
//
// One work unit = (query row r, shard d, split s): all H <= 128 heads of the
// row (the MMA M dimension) against the split's shard tokens.  A unit runs on
// a cluster of two CTAs.  CTA c owns half of the 576 latent dims:
//   c = 0: dims [0, 256) and [512, 544);  c = 1: dims [256, 512) and [544, 576)
// and the 256 value dims it owns are a subset of them, so every KV byte is
// loaded from HBM exactly once, by exactly one CTA.  Per 32-token tile:
//   producer warp  TMA-loads the CTA's 288 dims of the tile's tokens
//                  (4 x 64-dim 128B-swizzled boxes + 1 x 32-dim 64B-swizzled
//                  box per group of rows of one block) into a stage ring;
//   MMA warp       S_c = Q_c K_c^T with Q_c (128 x 288 bf16) resident in TMEM
//                  (18 tcgen05.mma, M=128 N=32 K=16), then, one tile behind,
//                  O_c += P V_c (P bf16 in TMEM, V_c the same smem tiles read
//                  MN-major, N=256 K=16);
//   softmax warps  thread = head = TMEM lane: swap the fp32 partial S with the
//                  peer CTA (one 16 KB DSMEM bulk copy each way), add, online
//                  softmax in base 2 with a lazy rescale (the running max is
//                  only moved when it grows by more than 2^8), P -> TMEM
//                  as bf16 while the normaliser sums the fp32 weights.
// Both CTAs hold the same S, so they take the same softmax decisions; each
// writes its 256 output dims, CTA 0 the LSE.  No tensor-core work is
// duplicated.  Every wait is bounded (a timeout sets DCP_DEVERR_TIMEOUT and
// ends the unit).
#include "dcp_kernels.h"
#include "dcp_sm100.cuh"

#include <cmath>
#include <cstring>

#include <cuda.h>

namespace dcp {
namespace {

using namespace sm100;

constexpr int kTile = 32;        // tokens per tile (MMA N of S, K of PV)
constexpr int kStages = 8;       // KV stage ring
constexpr int kChunkBytes = kTile * 128;        // 32 rows x 64 bf16 (SW128)
constexpr int kHalfBytes = kTile * 64;          // 32 rows x 32 bf16 (SW64)
constexpr int kStageBytes = 4 * kChunkBytes + kHalfBytes;  // 18 KB: 288 dims x 32 tokens
constexpr int kXBytes = 128 * kTile * 4;        // partial S exchange: 128 rows x 32 fp32
constexpr int kThreads = 192;    // warps 0-3 softmax, 4 MMA, 5 TMA producer
constexpr float kRescaleLog2 = 8.0f;

// TMEM columns
constexpr uint32_t kColQ = 0;     // 144 columns: Q_c, 288 bf16 per lane
constexpr uint32_t kColS = 160;   // 2 x 32 columns: partial S / P (bf16, first 16)
constexpr uint32_t kColO = 256;   // 256 columns: O_c
constexpr uint32_t kTmemCols = 512;

struct __align__(8) Bars {
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_free[2], p_full[2];
  uint64_t pv_done;
  uint64_t xfull[2], xfree[2];
  uint64_t xready[2], xcons[2];  // all 128 softmax threads wrote xout / read xin
  uint64_t o_final;              // last PV complete
  uint64_t fin;
  uint32_t mask[kStages];
  uint32_t tmem;
  int32_t abort;
};

constexpr int kOffStages = 0;
constexpr int kOffXout = kStages * kStageBytes;
constexpr int kOffXin = kOffXout + 2 * kXBytes;
constexpr int kOffBars = kOffXin + 2 * kXBytes;
constexpr int kSmemBytes = kOffBars + static_cast<int>(sizeof(Bars)) + 1024;  // + alignment slack

struct TcParams {
  int32_t mode_whole_blocks;  // 0: runs of I inside blocks (block_size % (D*I) == 0); 1: I % block_size == 0
  int32_t rows_per_box;       // R
  int32_t tok_per_block;      // tokens of one shard in one block (mode 0)
};

__device__ __forceinline__ void report(int32_t* dev_error, uint32_t bits) {
  if (dev_error) atomicOr(dev_error, static_cast<int32_t>(bits));
}

__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm128, const __grid_constant__ CUtensorMap tm64,
                 DecodeArgs a, TcParams tp) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  Bars& bar = *reinterpret_cast<Bars*>(smem + kOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();
  const uint32_t peer = cta ^ 1u;

  const int64_t unit = blockIdx.x >> 1;
  const int per_row = a.D * a.plan.splits;
  const int r = static_cast<int>(unit / per_row);
  const int d = static_cast<int>((unit % per_row) / a.plan.splits);
  const int s = static_cast<int>(unit % a.plan.splits);

  const RowInfo ri = resolve_row(a.seq_lens, a.qsl, a.B, r, a.max_seq_len, a.max_q_len);
  if (ri.err && threadIdx.x == 0 && cta == 0 && d == 0 && s == 0) report(a.dev_error, ri.err);
  const int32_t n_local = ri.padding ? 0 : local_len(ri.L, d, a.D, a.I);
  const int32_t lo = s * a.plan.chunk;
  const int32_t hi = min(n_local, lo + a.plan.chunk);
  const int ntiles = lo < hi ? (hi - lo + kTile - 1) / kTile : 0;
  const int64_t pair0 = ((static_cast<int64_t>(s) * a.D + d) * a.T + r) * a.H;

  if (ntiles == 0) {
    // empty shard / split or padding row: masked at the source, no KV read
    if (warp < 4) {
      const int h = threadIdx.x;
      if (h < a.H) {
        float* o = a.O_dst + (pair0 + h) * kLatent + 256 * cta;
        for (int i = 0; i < 64; ++i) reinterpret_cast<float4*>(o)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (cta == 0) a.lse_dst[pair0 + h] = -INFINITY;
      }
    }
    return;
  }

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&bar.kv_full[i], 1); mbar_init(&bar.kv_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.s_free[i], 1);
      mbar_init(&bar.p_full[i], 128);
      mbar_init(&bar.xfull[i], 1);
      mbar_init(&bar.xfree[i], 1);
      mbar_init(&bar.xready[i], 128);
      mbar_init(&bar.xcons[i], 128);
    }
    mbar_init(&bar.pv_done, 1);
    mbar_init(&bar.o_final, 1);
    mbar_init(&bar.fin, 1);
    bar.abort = 0;
    fence_mbar_init();
    // both exchange slots start free: expect the peer's first two copies
    mbar_arrive_expect_tx(&bar.xfull[0], kXBytes);
    mbar_arrive_expect_tx(&bar.xfull[1], kXBytes);
  }
  if (warp == 4) {
    tmem_alloc(&bar.tmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 5 && lane == 0) {
    tma_prefetch_desc(&tm128);
    tma_prefetch_desc(&tm64);
  }
  // Q_c -> TMEM (softmax warps; thread = head = lane)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bar.tmem;
  if (warp < 4) {
    const int h = threadIdx.x;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    const uint4* qrow = reinterpret_cast<const uint4*>(a.q + static_cast<int64_t>(r) * a.q_stride_tok +
                                                       static_cast<int64_t>(h < a.H ? h : 0) * kKDim);
    for (int i = 0; i < 4; ++i) {
      uint32_t v[32];
      const int dim0 = 256 * cta + 64 * i;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint4 x = h < a.H ? __ldg(qrow + dim0 / 8 + k) : make_uint4(0u, 0u, 0u, 0u);
        v[4 * k] = x.x; v[4 * k + 1] = x.y; v[4 * k + 2] = x.z; v[4 * k + 3] = x.w;
      }
      tmem_st32(lane_addr + kColQ + 32 * i, v);
    }
    {
      uint32_t v[16];
      const int dim0 = 512 + 32 * cta;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 x = h < a.H ? __ldg(qrow + dim0 / 8 + k) : make_uint4(0u, 0u, 0u, 0u);
        v[4 * k] = x.x; v[4 * k + 1] = x.y; v[4 * k + 2] = x.z; v[4 * k + 3] = x.w;
      }
      tmem_st16(lane_addr + kColQ + 128, v);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // peer's barriers initialised and armed before any remote operation
  tc_fence_after();

  const int32_t* trow = a.block_table + static_cast<int64_t>(ri.b) * a.bt_stride;
  const uint32_t smem_base = smem_u32(smem);
  int xdone = 0;  // softmax: exchange tiles received from the peer

  if (warp == 5) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int R = tp.rows_per_box;
      const int nbox = kTile / R;
      const int runs = a.I / a.block_size;  // mode 1: blocks per run
      int last[kStages];
      for (int i = 0; i < kStages; ++i) last[i] = -1;
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % kStages;
        if (!mbar_wait(&bar.kv_empty[st], ((j / kStages) & 1) ^ 1)) {
          report(a.dev_error, DCP_DEVERR_TIMEOUT);
          atomicExch(&bar.abort, 1);
          break;
        }
        if (*reinterpret_cast<volatile int32_t*>(&bar.abort)) break;
        const int32_t j0 = lo + j * kTile;
        uint32_t mask = 0;
        int loaded = 0;
        unsigned char* sbuf = smem + kOffStages + st * kStageBytes;
        int32_t coords[8][2];  // (k coordinate, physical block) per box
        for (int bx = 0; bx < nbox; ++bx) {
          const int32_t l0 = j0 + bx * R;
          coords[bx][0] = -1;
          if (l0 >= hi) continue;
          int32_t lblk, kc;
          if (tp.mode_whole_blocks) {
            const int32_t lb = l0 / a.block_size, o = l0 % a.block_size;
            lblk = (lb / runs) * (a.D * runs) + d * runs + lb % runs;
            kc = o;
          } else {
            lblk = l0 / tp.tok_per_block;
            kc = (l0 % tp.tok_per_block) / a.I;
          }
          const int32_t blk = __ldg(trow + lblk);
          if (blk < 0 || blk >= a.num_blocks) {
            report(a.dev_error, DCP_DEVERR_BAD_BLOCK);
            continue;
          }
          coords[bx][0] = kc;
          coords[bx][1] = blk;
          const int nvalid = min(R, hi - l0);
          mask |= (nvalid >= 32 ? 0xffffffffu : ((1u << nvalid) - 1u)) << (bx * R);
          ++loaded;
        }
        bar.mask[st] = mask;
        last[st] = j;
        mbar_arrive_expect_tx(&bar.kv_full[st], static_cast<uint32_t>(loaded * R * (4 * 128 + 64)));
        const int32_t dsel = tp.mode_whole_blocks ? 0 : d;
        for (int bx = 0; bx < nbox; ++bx) {
          if (coords[bx][0] < 0) continue;
          const int32_t kc = coords[bx][0], blk = coords[bx][1];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            tma_load_5d(sbuf + i * kChunkBytes + bx * R * 128, &tm128, &bar.kv_full[st],
                        256 * static_cast<int32_t>(cta) + 64 * i, 0, dsel, kc, blk);
          tma_load_5d(sbuf + 4 * kChunkBytes + bx * R * 64, &tm64, &bar.kv_full[st],
                      512 + 32 * static_cast<int32_t>(cta), 0, dsel, kc, blk);
        }
      }
      // every load this CTA issued has landed before its shared memory goes away
      for (int i = 0; i < kStages; ++i)
        if (last[i] >= 0) mbar_wait(&bar.kv_full[i], (last[i] / kStages) & 1);
    }
  } else if (warp == 4) {
    // ----------------------------------------------------------------- MMA
    const uint32_t id_s = idesc_bf16(128, kTile, 0, 0);
    const uint32_t id_o = idesc_bf16(128, 256, 0, 1);
    bool ok = true;
    for (int j = 0; j <= ntiles && ok; ++j) {
      if (j < ntiles) {
        const int st = j % kStages, b = j & 1;
        ok = mbar_wait(&bar.kv_full[st], (j / kStages) & 1) && mbar_wait(&bar.s_free[b], ((j >> 1) & 1) ^ 1);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint32_t mask = bar.mask[st];
        if (mask != 0xffffffffu) {
          // rows not loaded (tail, bad block) or past the split: zero them so
          // that P = 0 never meets a NaN/Inf value row
          unsigned char* sbuf = smem + kOffStages + st * kStageBytes;
          for (int row = 0; row < kTile; ++row) {
            if (mask & (1u << row)) continue;
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<uint32_t*>(sbuf + i * kChunkBytes + row * 128)[lane] = 0u;
            if (lane < 16) reinterpret_cast<uint32_t*>(sbuf + 4 * kChunkBytes + row * 64)[lane] = 0u;
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sb = smem_base + kOffStages + st * kStageBytes;
          const uint32_t dS = tbase + kColS + 32 * b;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            mma_ts(dS, tbase + kColQ + 8 * k,
                   smem_desc(sb + (k >> 2) * kChunkBytes + (k & 3) * 32, 16, 1024, kSwizzle128B), id_s, k > 0);
#pragma unroll
          for (int k = 0; k < 2; ++k)
            mma_ts(dS, tbase + kColQ + 128 + 8 * k, smem_desc(sb + 4 * kChunkBytes + k * 32, 16, 512, kSwizzle64B),
                   id_s, 1);
          mma_commit(&bar.s_full[b]);
        }
        __syncwarp();
      }
      if (j >= 1) {
        const int jp = j - 1, bp = jp & 1, stp = jp % kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar.p_full[bp], (jp >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sb = smem_base + kOffStages + stp * kStageBytes;
#pragma unroll
          for (int k = 0; k < 2; ++k)
            mma_ts(tbase + kColO, tbase + kColS + 32 * bp + 8 * k,
                   smem_desc(sb + 2048 * k, kChunkBytes, 1024, kSwizzle128B), id_o, (jp > 0 || k > 0) ? 1u : 0u);
          mma_commit(&bar.kv_empty[stp]);
          mma_commit(&bar.s_free[bp]);
          mma_commit(&bar.pv_done);
          if (jp == ntiles - 1) mma_commit(&bar.o_final);
        }
        __syncwarp();
      }
    }
    if (!ok) {
      report(a.dev_error, DCP_DEVERR_TIMEOUT);
      atomicExch(&bar.abort, 1);
    }
    // all issued MMAs complete before TMEM is released
    if (lane == 0) mma_commit(&bar.fin);
    __syncwarp();
    mbar_wait(&bar.fin, 0);
  } else {
    // ------------------------------------------------------------- softmax
    const int h = threadIdx.x;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl2 = a.scale * kLog2e;
    float m_used = -INFINITY, l_sum = 0.f;
    unsigned char* xout = smem + kOffXout;
    unsigned char* xin = smem + kOffXin;
    const int sw = h & 7;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1, st = j % kStages, n = j >> 1;
      ok = mbar_wait(&bar.s_full[b], n & 1) && mbar_wait(&bar.kv_full[st], (j / kStages) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(lane_addr + kColS + 32 * b, sr);
      tmem_wait_ld();
      const uint32_t mask = bar.mask[st];
      // swap partial scores with the peer: xout[b] is free once the peer has
      // consumed tile j-2 (which also means that copy has finished reading it)
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(&bar.xfree[b], (n & 1) ^ 1));
      if (!ok) break;
      float4* xo = reinterpret_cast<float4*>(xout + b * kXBytes + h * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        xo[c ^ sw] = make_float4(__uint_as_float(sr[4 * c]), __uint_as_float(sr[4 * c + 1]),
                                 __uint_as_float(sr[4 * c + 2]), __uint_as_float(sr[4 * c + 3]));
      fence_proxy_async_smem();
      mbar_arrive(&bar.xready[b]);
      if (h == 0) {
        ok = mbar_wait(&bar.xready[b], n & 1);
        if (ok)
          bulk_copy_to_peer(map_peer(smem_base + kOffXin + b * kXBytes, peer), xout + b * kXBytes, kXBytes,
                            map_peer(smem_u32(&bar.xfull[b]), peer));
      }
      __syncwarp();
      ok = __all_sync(0xffffffffu, ok && mbar_wait_cluster(&bar.xfull[b], n & 1));
      if (!ok) break;
      ++xdone;
      const float4* xi = reinterpret_cast<const float4*>(xin + b * kXBytes + h * 128);
      float sc[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 p = xi[c ^ sw];
        sc[4 * c] = __uint_as_float(sr[4 * c]) + p.x;
        sc[4 * c + 1] = __uint_as_float(sr[4 * c + 1]) + p.y;
        sc[4 * c + 2] = __uint_as_float(sr[4 * c + 2]) + p.z;
        sc[4 * c + 3] = __uint_as_float(sr[4 * c + 3]) + p.w;
      }
      mbar_arrive(&bar.xcons[b]);
      if (h == 0) {
        // once all 128 rows are read: re-arm for tile j + 2, then let the peer send it
        ok = mbar_wait(&bar.xcons[b], n & 1);
        if (ok) {
          mbar_arrive_expect_tx(&bar.xfull[b], kXBytes);
          mbar_arrive_remote(map_peer(smem_u32(&bar.xfree[b]), peer));
        }
      }
      __syncwarp();
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // online softmax (base 2), masked tokens get weight 0 by selection
      float tmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        sc[i] = (mask >> i) & 1u ? sc[i] * sl2 : -INFINITY;
        tmax = fmaxf(tmax, sc[i]);
      }
      const bool grow = m_used == -INFINITY ? (tmax != -INFINITY) : (tmax > m_used + kRescaleLog2);
      float alpha = 1.f;
      float m_new = m_used;
      if (grow) {
        m_new = tmax;
        if (m_used != -INFINITY) alpha = exp2f(m_used - m_new);
      }
      const bool need_rescale = grow && m_used != -INFINITY;
      if (__any_sync(0xffffffffu, need_rescale)) {
        // O holds PV(0..j-1): wait for PV(j-1), then scale this warp's rows
        ok = __all_sync(0xffffffffu, mbar_wait(&bar.pv_done, (j - 1) & 1));
        if (!ok) break;
        tc_fence_after();
        for (int c = 0; c < 8; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kColO + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(lane_addr + kColO + 32 * c, o);
        }
        tmem_wait_st();
      }
      l_sum *= alpha;
      m_used = m_new;
      uint32_t pk[16];
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        // masked tokens are exactly -inf: weight 0 (also when nothing is live yet)
        const float p0 = sc[2 * i] == -INFINITY ? 0.f : exp2f(sc[2 * i] - m_used);
        const float p1 = sc[2 * i + 1] == -INFINITY ? 0.f : exp2f(sc[2 * i + 1] - m_used);
        __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);  // P feeds the PV MMA in bf16
        psum += p0 + p1;                                     // l (hence the LSE) stays fp32
        pk[i] = *reinterpret_cast<uint32_t*>(&pb);
      }
      l_sum += psum;
      tmem_st16(lane_addr + kColS + 32 * b, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar.p_full[b]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar.o_final, 0));
    if (ok) ok = !__any_sync(0xffffffffu, *reinterpret_cast<volatile int32_t*>(&bar.abort) != 0);
    if (!ok) {
      report(a.dev_error, DCP_DEVERR_TIMEOUT);
      atomicExch(&bar.abort, 1);
    } else {
      tc_fence_after();
      const int64_t pair = pair0 + h;
      const bool live = l_sum > 0.f;
      const float inv = live ? 1.f / l_sum : 0.f;
      float* orow = a.O_dst + pair * kLatent + 256 * cta;
      for (int c = 0; c < 8; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + kColO + 32 * c, o);
        tmem_wait_ld();
        if (h < a.H) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(orow + 32 * c)[i] =
                make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                            __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
        }
      }
      if (h < a.H && cta == 0) a.lse_dst[pair] = live ? (m_used + log2f(l_sum)) * kLn2 : -INFINITY;
    }
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  const bool aborted = *reinterpret_cast<volatile int32_t*>(&bar.abort) != 0;
  __syncthreads();
  cluster_sync();  // the peer has issued everything it will send here
  if (aborted && threadIdx.x == 0) {
    // a failed unit may have left one of the peer's copies in flight into
    // xin: give each slot's next phase a short bounded wait before exiting
    for (int b = 0; b < 2; ++b) {
      const int received = (xdone + 1 - b) / 2;
      mbar_wait_cluster(&bar.xfull[b], received & 1, 1u << 16);
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool tc_params(const DecodeArgs& a, TcParams& tp) {
  if (a.H > 128) return false;
  const int bs = a.block_size, D = a.D, I = a.I;
  if (I % bs == 0) {
    const int R = bs < kTile ? bs : kTile;
    if (R < 4 || kTile % R || bs % R) return false;
    tp.mode_whole_blocks = 1;
    tp.rows_per_box = R;
    tp.tok_per_block = bs;
    return true;
  }
  if (bs % (D * I) == 0) {
    const int tpb = bs / D;
    const int R = tpb < kTile ? tpb : kTile;
    if (R < 4 || kTile % R || tpb % R || R % I) return false;
    tp.mode_whole_blocks = 0;
    tp.rows_per_box = R;
    tp.tok_per_block = tpb;
    return true;
  }
  return false;
}

}  // namespace

bool decode_tc_supported(const DecodeArgs& a) {
  TcParams tp;
  return tc_params(a, tp) && (a.plan.chunk % kTile) == 0;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
  TcParams tp;
  if (!tc_params(a, tp)) return cudaErrorInvalidValue;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  // 5-D view of the cache: [576 dims][run of I][shard][run index][block]
  // (mode 1: [576][1][1][block_size][block]); box = 64 (or 32) dims x R rows.
  const int bs = a.block_size;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5], es[5] = {1, 1, 1, 1, 1};
  dims[0] = kKDim;
  if (tp.mode_whole_blocks) {
    dims[1] = 1; dims[2] = 1; dims[3] = static_cast<cuuint64_t>(bs);
    strides[0] = kKDim * 2; strides[1] = kKDim * 2; strides[2] = kKDim * 2;
    box[1] = 1; box[2] = 1; box[3] = static_cast<cuuint32_t>(tp.rows_per_box);
  } else {
    dims[1] = static_cast<cuuint64_t>(a.I);
    dims[2] = static_cast<cuuint64_t>(a.D);
    dims[3] = static_cast<cuuint64_t>(bs / (a.D * a.I));
    strides[0] = kKDim * 2;
    strides[1] = static_cast<cuuint64_t>(kKDim) * 2 * a.I;
    strides[2] = static_cast<cuuint64_t>(kKDim) * 2 * a.I * a.D;
    box[1] = static_cast<cuuint32_t>(a.I); box[2] = 1; box[3] = static_cast<cuuint32_t>(tp.rows_per_box / a.I);
  }
  dims[4] = static_cast<cuuint64_t>(a.num_blocks);
  strides[3] = static_cast<cuuint64_t>(kKDim) * 2 * bs;
  box[4] = 1;
  CUtensorMap m128, m64;
  void* base = const_cast<__nv_bfloat16*>(a.kv);
  box[0] = 64;
  if (enc(&m128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  box[0] = 32;
  if (enc(&m64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t units = static_cast<int64_t>(a.T) * a.D * a.plan.splits;
  if (2 * units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * units));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel, m128, m64, a, tp);
}

}  // namespace dcp
