// Tensor-core split-KV MLA decode for sm_103a (tcgen05 + TMEM + TMA + DSMEM).
//
// One work unit = (query row r, shard d, split s): all H <= 128 heads of the
// row (the MMA M dimension) against the split's shard tokens.  A unit runs on
// a cluster of two CTAs that split the 576 latent dims by 64-dim chunks:
//   CTA 0: chunks 0-3 = dims [0, 256)        (its value dims [0, 256))
//   CTA 1: chunks 4-8 = dims [256, 576)      (its value dims [256, 512) and
//                                             the 64 rope dims)
// so every KV byte is loaded from HBM exactly once, by exactly one CTA, as a
// single run of consecutive chunks.  Per 32-token tile:
//   producers (2)  TMA-load the CTA's chunks of the tile's tokens into a
//                  stage ring (alternate tiles).  A 5-D tensor map whose chunk dimension comes
//                  after the row dimensions lets one box carry all of the
//                  CTA's chunks for a group of rows of one block (a box costs
//                  tens of cycles to issue whatever it carries);
//   S warps (3)    S(j) = Q_c K_c^T with Q_c (128 rows x 256 or 320 dims,
//                  bf16) resident in TMEM: 16 or 20 tcgen05.mma (M=128 N=32
//                  K=16) into S buffer j mod 3, issued by warp 6 + (j mod 3)
//                  (a tcgen05.mma occupies its issuing thread far longer than
//                  an N=32 product takes, so issue is spread over warps);
//   PV warp        O_c += P(j) V_c in tile order (P bf16 in TMEM, V_c = the
//                  CTA's first four chunks of the same tiles read MN-major,
//                  N=256 K=16);
//   softmax warps  thread = head = TMEM lane: ship the fp32 partial S of tile
//                  j+1 to the peer CTA (a 4 KB DSMEM bulk copy per warp,
//                  completing on the peer's mbarrier) before working on tile
//                  j, add the peer's partial of tile j, online softmax in
//                  base 2 with a lazy rescale (the running max only moves
//                  when it grows by more than 2^8), P -> TMEM as bf16 while
//                  the normaliser sums the fp32 weights.
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

constexpr int kTile = 32;                        // tokens per tile (MMA N of S, K of PV)
constexpr int kStages = 6;                       // KV stage ring
constexpr int kSBuf = 3;                         // S buffers in TMEM = exchange slots in smem
constexpr int kChunkBytes = kTile * 128;         // 32 rows x 64 bf16, 128B-swizzled
constexpr int kMaxChunks = 5;                    // chunks one CTA loads (CTA 1)
constexpr int kStageBytes = kMaxChunks * kChunkBytes;  // 20 KB
constexpr int kXBytes = 128 * kTile * 4;         // partial S exchange: 128 rows x 32 fp32
constexpr int kXWarpBytes = kXBytes / 4;         // one softmax warp's 32 rows
constexpr int kThreads = 320;                    // warps 0-3 softmax, 4 PV, 5 + 9 producers, 6-8 S
constexpr float kRescaleLog2 = 8.0f;

// TMEM columns
constexpr uint32_t kColQ = 0;     // up to 160 columns: Q_c, 2 bf16 per column
constexpr uint32_t kColS = 160;   // 3 x 32 columns: partial S / P (bf16, first 16)
constexpr uint32_t kColO = 256;   // 256 columns: O_c
constexpr uint32_t kTmemCols = 512;

struct __align__(8) Bars {
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[kSBuf], s_free[kSBuf], p_full[kSBuf];
  uint64_t xfull[kSBuf], xfree[kSBuf];  // 4 arrivals each (one per softmax warp)
  uint64_t pv_done[2];                  // PV(j) completes phase j / 2 of pv_done[j & 1]
  uint64_t o_final;                     // last PV complete
  uint64_t fin[1 + kSBuf];              // each issuing warp's MMAs complete
  uint32_t mask[kStages];
  uint32_t tmem;
  int32_t abort;
};

constexpr int kOffStages = 0;
constexpr int kOffXin = kStages * kStageBytes;
constexpr int kOffXout = kOffXin + kSBuf * kXBytes;
constexpr int kOffBars = kOffXout + kSBuf * kXBytes;
constexpr int kSmemBytes = kOffBars + static_cast<int>(sizeof(Bars)) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory per CTA");
static_assert(kStages % 2 == 0, "the two producer warps own alternate stages");

// How a tile's 32 shard tokens reach shared memory.  R consecutive shard
// tokens lie in one block.  Layout kinds (Rb rows per box, Cb chunks per box):
//   0: Rb = 8,  Cb = all: group-major stage (8-row groups nch KB apart,
//                          chunk stride 1 KB)
//   1: Rb = 32, Cb = all: chunk-major stage (chunk stride 4 KB, groups 1 KB)
//   2: Rb = R,  Cb = 1:   chunk-major stage, one box per chunk (an 8-row
//                          group would split a run of the interleave)
struct TcParams {
  int32_t mode_whole_blocks;  // 0: runs of I inside blocks (block_size % (D*I) == 0); 1: I % block_size == 0
  int32_t rows_per_box;       // R
  int32_t tok_per_block;      // tokens of one shard in one block (mode 0)
  int32_t run;                // rows of one interleave run inside a box (I in mode 0, 1 in mode 1)
  int32_t kind;               // layout kind above
  int32_t box_rows;           // Rb
};

__device__ __forceinline__ void report(int32_t* dev_error, uint32_t bits) {
  if (dev_error) atomicOr(dev_error, static_cast<int32_t>(bits));
}

__device__ __forceinline__ bool aborted(Bars& bar) { return *reinterpret_cast<volatile int32_t*>(&bar.abort) != 0; }

__device__ __forceinline__ void set_abort(Bars& bar, int32_t* dev_error) {
  report(dev_error, DCP_DEVERR_TIMEOUT);
  atomicExch(&bar.abort, 1);
}

__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                 DecodeArgs a, TcParams tp) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  Bars& bar = *reinterpret_cast<Bars*>(smem + kOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();
  const uint32_t peer = cta ^ 1u;
  const int nch = 4 + static_cast<int>(cta);     // chunks this CTA owns
  const int chunk0 = 4 * static_cast<int>(cta);  // first of them
  // stage layout of this CTA (see TcParams)
  const int chunk_stride = tp.kind == 0 ? 1024 : kChunkBytes;
  const int group_stride = tp.kind == 0 ? 1024 * nch : 1024;
  const CUtensorMap* tmap = cta == 0 ? &tm0 : &tm1;

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
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.s_free[i], 1);
      mbar_init(&bar.p_full[i], 4);  // one arrival per softmax warp
      mbar_init(&bar.xfull[i], 4);
      mbar_init(&bar.xfree[i], 4);
    }
    mbar_init(&bar.pv_done[0], 1);
    mbar_init(&bar.pv_done[1], 1);
    mbar_init(&bar.o_final, 1);
    for (int i = 0; i < 1 + kSBuf; ++i) mbar_init(&bar.fin[i], 1);
    bar.abort = 0;
    fence_mbar_init();
    // every exchange slot starts free: expect the peer's first partials
    // (four 4 KB copies per slot, one per peer softmax warp)
    for (int i = 0; i < kSBuf; ++i)
      for (int w = 0; w < 4; ++w) mbar_arrive_expect_tx(&bar.xfull[i], kXWarpBytes);
  }
  if (warp == 4) {
    tmem_alloc(&bar.tmem, kTmemCols);
    tmem_relinquish();
  }
  if ((warp == 5 || warp == 9) && lane == 0) tma_prefetch_desc(tmap);
  // Q_c -> TMEM (softmax warps; thread = head = lane): dim k of the CTA's
  // chunks goes to column k / 2 (low half = even k)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bar.tmem;
  if (warp < 4) {
    const int h = threadIdx.x;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    const uint4* qrow = reinterpret_cast<const uint4*>(a.q + static_cast<int64_t>(r) * a.q_stride_tok +
                                                       static_cast<int64_t>(h < a.H ? h : 0) * kKDim);
    for (int i = 0; i < nch; ++i) {
      uint32_t v[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint4 x = h < a.H ? __ldg(qrow + (chunk0 + i) * 8 + k) : make_uint4(0u, 0u, 0u, 0u);
        v[4 * k] = x.x; v[4 * k + 1] = x.y; v[4 * k + 2] = x.z; v[4 * k + 3] = x.w;
      }
      tmem_st32(lane_addr + kColQ + 32 * i, v);
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

  if (warp == 5 || warp == 9) {
    // ----------------------------------------------------------- producers
    // Two warps (tiles j = p mod 2, hence disjoint stages, since kStages is
    // even): TMA issue occupies the issuing thread, so two issue in
    // parallel.  Per warp, the block ids of its own boxes g = 32k + lane are
    // fetched one batch ahead (a tile's boxes never straddle batches: 32 %
    // nbox == 0); lanes issue the tile's TMA boxes.
    const int p = warp == 5 ? 0 : 1;
    const int R = tp.rows_per_box;
    const int nbox = kTile / R;
    const int runs = a.I / a.block_size;  // mode 1: blocks per run
    const int32_t dsel = tp.mode_whole_blocks ? 0 : d * a.I;  // first row of shard d in a run group
    const int Rb = tp.box_rows, nsub = kTile / Rb, npc = tp.kind == 2 ? nch : 1;
    auto box_k = [&](int32_t l0) -> int32_t {
      return tp.mode_whole_blocks ? l0 % a.block_size : (l0 % tp.tok_per_block) / a.I;
    };
    auto fetch = [&](int k) -> int32_t {  // -2: past the split, -1: bad block id
      const int g = 32 * k + lane;                            // this warp's box g
      const int jj = p + 2 * (g / nbox);                      // its tile
      const int32_t l0 = lo + (jj * nbox + g % nbox) * R;     // its first shard token
      if (l0 >= hi) return -2;
      int32_t lblk;
      if (tp.mode_whole_blocks) {
        const int32_t lb = l0 / a.block_size;
        lblk = (lb / runs) * (a.D * runs) + d * runs + lb % runs;
      } else {
        lblk = l0 / tp.tok_per_block;
      }
      const int32_t blk = __ldg(trow + lblk);
      return (blk < 0 || blk >= a.num_blocks) ? -1 : blk;
    };
    int32_t cur = fetch(0), nxt = fetch(1);
    int kcur = 0;
    int last[kStages];
    for (int i = 0; i < kStages; ++i) last[i] = -1;
    for (int m = 0; p + 2 * m < ntiles; ++m) {
      const int j = p + 2 * m;
      const int st = j % kStages;
      bool ok = lane == 0 ? mbar_wait(&bar.kv_empty[st], ((j / kStages) & 1) ^ 1) : true;
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) { if (lane == 0) set_abort(bar, a.dev_error); break; }
      if (__any_sync(0xffffffffu, aborted(bar))) break;
      const int g0 = m * nbox;  // this warp's first box of the tile
      if ((g0 >> 5) != kcur) { cur = nxt; ++kcur; nxt = fetch(kcur + 1); }
      // lane bx < nbox owns R-row box bx of this tile
      const int32_t blk = __shfl_sync(0xffffffffu, cur, (g0 + lane) & 31);
      const bool mine = lane < nbox;
      const int32_t l0 = lo + (j * nbox + lane) * R;
      if (mine && blk == -1) report(a.dev_error, DCP_DEVERR_BAD_BLOCK);
      const bool valid = mine && blk >= 0;
      const int nvalid = valid ? min(R, hi - l0) : 0;
      const uint32_t bits = valid ? ((nvalid >= 32 ? 0xffffffffu : ((1u << nvalid) - 1u)) << (lane * R)) : 0u;
      const uint32_t mask = __reduce_or_sync(0xffffffffu, bits);
      const int loaded = __popc(__ballot_sync(0xffffffffu, valid));
      if (lane == 0) {
        bar.mask[st] = mask;
        mbar_arrive_expect_tx(&bar.kv_full[st], static_cast<uint32_t>(loaded * R * nch * 128));
      }
      last[st] = j;
      __syncwarp();
      unsigned char* sbuf = smem + kOffStages + st * kStageBytes;
      // (sub-box, piece) pairs q = lane, lane + 32
      for (int q0 = 0; q0 < nsub * npc; q0 += 32) {
        const int q = q0 + lane;
        const int sb = (q / npc) & 7, piece = q % npc;
        const int bx = (sb * Rb) / R;  // the R-row box (block) holding this sub-box
        const int32_t b_blk = __shfl_sync(0xffffffffu, blk, bx);
        const bool b_valid = __shfl_sync(0xffffffffu, valid ? 1 : 0, bx) != 0;
        if (q < nsub * npc && b_valid) {
          const int32_t kc = box_k(lo + (j * nbox + bx) * R) + ((sb * Rb) % R) / tp.run;
          unsigned char* dst = tp.kind == 0 ? sbuf + sb * group_stride
                             : tp.kind == 1 ? sbuf
                                            : sbuf + piece * kChunkBytes + sb * Rb * 128;
          tma_load_5d(dst, tmap, &bar.kv_full[st], 0, dsel, kc, chunk0 + piece, b_blk);
        }
      }
    }
    // every load this CTA issued has landed before its shared memory goes away
    if (lane == 0)
      for (int i = 0; i < kStages; ++i)
        if (last[i] >= 0) mbar_wait(&bar.kv_full[i], (last[i] / kStages) & 1);
  } else if (warp >= 6) {
    // ------------------------------------------------------- S MMA issuers
    // warp 6+i owns S buffer i and tiles j = i (mod 3)
    const int b = warp - 6;
    const uint32_t id_s = idesc_bf16(128, kTile, 0, 0);
    const uint64_t dk = smem_desc(smem_base + kOffStages, 16, group_stride, kSwizzle128B);
    const uint32_t dS = tbase + kColS + 32 * b;
    const int ksteps = 4 * nch;
    bool ok = true;
    for (int j = b; j < ntiles; j += kSBuf) {
      const int st = j % kStages, u = j / kSBuf;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.kv_full[st], (j / kStages) & 1) &&
                                       mbar_wait(&bar.s_free[b], (u & 1) ^ 1));
      if (!ok) break;
      const uint32_t mask = bar.mask[st];
      if (mask != 0xffffffffu) {
        // rows not loaded (tail, bad block): zero them so that P = 0 never
        // meets a NaN/Inf value row
        unsigned char* sbuf = smem + kOffStages + st * kStageBytes;
        for (int row = 0; row < kTile; ++row) {
          if (mask & (1u << row)) continue;
          for (int i = 0; i < nch; ++i)
            reinterpret_cast<uint32_t*>(sbuf + i * chunk_stride + (row >> 3) * group_stride + (row & 7) * 128)[lane] =
                0u;
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
        const uint64_t so = static_cast<uint64_t>((st * kStageBytes) >> 4);
        for (int k = 0; k < ksteps; ++k)
          mma_ts(dS, tbase + kColQ + 8 * k, dk + so + (((k >> 2) * chunk_stride + (k & 3) * 32) >> 4), id_s, k > 0);
        mma_commit(&bar.s_full[b]);
      }
      __syncwarp();
    }
    if (!ok) set_abort(bar, a.dev_error);
    if (lane == 0) mma_commit(&bar.fin[1 + b]);
    __syncwarp();
    mbar_wait(&bar.fin[1 + b], 0);
  } else if (warp == 4) {
    // -------------------------------------------------------- PV MMA issuer
    // O accumulates across tiles, so PV(j) is issued in order by one thread.
    // V_c (the CTA's first four chunks) is the MN-major B operand: N (value
    // dims) atoms = chunks, K (tokens) in 8-row groups.
    const uint32_t id_o = idesc_bf16(128, 256, 0, 1);
    const uint64_t dv = smem_desc(smem_base + kOffStages, chunk_stride, group_stride, kSwizzle128B);
    bool ok = true;
    for (int jp = 0; jp < ntiles; ++jp) {
      const int st = jp % kStages, b = jp % kSBuf;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.p_full[b], (jp / kSBuf) & 1));
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t so = static_cast<uint64_t>((st * kStageBytes) >> 4);
#pragma unroll
        for (int k = 0; k < 2; ++k)
          mma_ts(tbase + kColO, tbase + kColS + 32 * b + 8 * k, dv + so + ((2 * group_stride * k) >> 4), id_o,
                 (jp > 0 || k > 0) ? 1u : 0u);
        mma_commit(&bar.kv_empty[st]);
        mma_commit(&bar.s_free[b]);
        mma_commit(&bar.pv_done[jp & 1]);
        if (jp == ntiles - 1) mma_commit(&bar.o_final);
      }
      __syncwarp();
    }
    if (!ok) set_abort(bar, a.dev_error);
    // all issued MMAs complete before TMEM is released
    if (lane == 0) mma_commit(&bar.fin[0]);
    __syncwarp();
    mbar_wait(&bar.fin[0], 0);
  } else {
    // ------------------------------------------------------------- softmax
    // Software-pipelined: the partial S of tile j+1 is shipped to the peer
    // before tile j's softmax, so the exchange latency hides behind a tile.
    const int h = threadIdx.x;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl2 = a.scale * kLog2e;
    float m_used = -INFINITY, l_sum = 0.f;
    const unsigned char* xin = smem + kOffXin;
    unsigned char* xout = smem + kOffXout;
    const int sw = h & 7;
    bool ok = true;
    // load own partial S(jj) from TMEM and ship it to the peer's slot
    auto send = [&](int jj, uint32_t (&sr)[32]) -> bool {
      const int b = jj % kSBuf, u = jj / kSBuf;
      if (!__all_sync(0xffffffffu, mbar_wait(&bar.s_full[b], u & 1))) return false;
      tc_fence_after();
      tmem_ld32(lane_addr + kColS + 32 * b, sr);
      tmem_wait_ld();
      // the peer's slot b (and our staging slot b) are free once the peer has
      // consumed tile jj - kSBuf
      if (!__all_sync(0xffffffffu, mbar_wait(&bar.xfree[b], (u & 1) ^ 1))) return false;
      float4* xo = reinterpret_cast<float4*>(xout + b * kXBytes + h * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        xo[c ^ sw] = make_float4(__uint_as_float(sr[4 * c]), __uint_as_float(sr[4 * c + 1]),
                                 __uint_as_float(sr[4 * c + 2]), __uint_as_float(sr[4 * c + 3]));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        bulk_copy_to_peer(map_peer(smem_base + kOffXin + b * kXBytes + warp * kXWarpBytes, peer),
                          xout + b * kXBytes + warp * kXWarpBytes, kXWarpBytes,
                          map_peer(smem_u32(&bar.xfull[b]), peer));
      return true;
    };
    uint32_t sr_cur[32], sr_nxt[32];
    ok = send(0, sr_cur);
    for (int j = 0; j < ntiles && ok; ++j) {
      const int b = j % kSBuf, st = j % kStages, u = j / kSBuf;
      if (j + 1 < ntiles && !send(j + 1, sr_nxt)) { ok = false; break; }
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.kv_full[st], (j / kStages) & 1) &&
                                       mbar_wait(&bar.xfull[b], u & 1));
      if (!ok) break;
      ++xdone;
      const uint32_t mask = bar.mask[st];
      const float4* xi = reinterpret_cast<const float4*>(xin + b * kXBytes + h * 128);
      float sc[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 p = xi[c ^ sw];
        sc[4 * c] = __uint_as_float(sr_cur[4 * c]) + p.x;
        sc[4 * c + 1] = __uint_as_float(sr_cur[4 * c + 1]) + p.y;
        sc[4 * c + 2] = __uint_as_float(sr_cur[4 * c + 2]) + p.z;
        sc[4 * c + 3] = __uint_as_float(sr_cur[4 * c + 3]) + p.w;
      }
      // online softmax (base 2); masked tokens get weight 0 by selection
      if (mask != 0xffffffffu) {
#pragma unroll
        for (int i = 0; i < 32; ++i) sc[i] = (mask >> i) & 1u ? sc[i] : -INFINITY;
      }
      // row max of the raw scores (scale > 0 commutes with max), as a tree
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = fmaxf(fmaxf(sc[4 * i], sc[4 * i + 1]), fmaxf(sc[4 * i + 2], sc[4 * i + 3]));
      const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
      const bool grow = m_used == -INFINITY ? (tmax != -INFINITY) : (tmax > m_used + kRescaleLog2);
      float alpha = 1.f;
      float m_new = m_used;
      if (grow) {
        m_new = tmax;
        if (m_used != -INFINITY) alpha = ex2_approx(m_used - m_new);
      }
      const bool need_rescale = grow && m_used != -INFINITY;
      if (__any_sync(0xffffffffu, need_rescale)) {
        // O holds PV(0..j-1): wait for PV(j-1), then scale this warp's rows.
        // pv_done[(j-1) & 1] sees PV(j-3) (complete: S(j) reused its
        // buffer), PV(j-1) and PV(j+1) (impossible before P(j)), so the
        // parity of phase (j-1)/2 is unambiguous.
        ok = __all_sync(0xffffffffu, mbar_wait(&bar.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1));
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
      // p = 2^(s * scale * log2e - m); masked (-inf) scores give exactly 0,
      // and nothing is live while m is still -inf
      const float nm = m_used == -INFINITY ? 0.f : -m_used;
      uint32_t pk[16];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = ex2_approx(fmaf(sc[2 * i], sl2, nm));
        const float p1 = ex2_approx(fmaf(sc[2 * i + 1], sl2, nm));
        __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);  // P feeds the PV MMA in bf16
        ps[i & 3] += p0 + p1;                                // l (hence the LSE) stays fp32
        pk[i] = *reinterpret_cast<uint32_t*>(&pb);
      }
      l_sum += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      tmem_st16(lane_addr + kColS + 32 * b, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar.p_full[b]);
        // this warp has consumed slot b (the values are in registers): expect
        // its next 4 KB and let the peer refill it
        mbar_arrive_expect_tx(&bar.xfull[b], kXWarpBytes);
        mbar_arrive_remote_relaxed(map_peer(smem_u32(&bar.xfree[b]), peer));
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) sr_cur[i] = sr_nxt[i];
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar.o_final, 0));
    if (ok) ok = !__any_sync(0xffffffffu, aborted(bar));
    if (!ok) {
      set_abort(bar, a.dev_error);
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
  const bool failed = aborted(bar);
  __syncthreads();
  cluster_sync();  // the peer has issued everything it will send here
  if (failed && threadIdx.x == 0) {
    // a failed unit may have left some of the peer's copies in flight into
    // its slots: give each slot's next phase a short bounded wait
    for (int b = 0; b < kSBuf; ++b) {
      const int received = xdone > b ? (xdone - 1 - b) / kSBuf + 1 : 0;
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
    tp.mode_whole_blocks = 1;
    tp.rows_per_box = bs < kTile ? bs : kTile;
    tp.tok_per_block = bs;
    tp.run = 1;
  } else if (bs % (D * I) == 0) {
    const int tpb = bs / D;
    tp.mode_whole_blocks = 0;
    tp.rows_per_box = tpb < kTile ? tpb : kTile;
    tp.tok_per_block = tpb;
    tp.run = I;
  } else {
    return false;
  }
  const int R = tp.rows_per_box;
  if (R < 4 || kTile % R || tp.tok_per_block % R || R % tp.run) return false;
  if (R == 32) {
    tp.kind = 1; tp.box_rows = 32;
  } else if (R >= 8 && 8 % tp.run == 0) {
    tp.kind = 0; tp.box_rows = 8;
  } else {
    tp.kind = 2; tp.box_rows = R;
  }
  return true;
}

}  // namespace

int decode_tc_resident_ctas() {
  // CTAs of the tensor-core decode that fit on the current device at once
  // (1 per SM by shared memory; clusters of two must sit in one GPC).
  static int cached_dev = -1, cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  if (dev == cached_dev) return cached;
  if (cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess) { cudaGetLastError(); return 0; }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, decode_tc_kernel, &cfg) != cudaSuccess || clusters <= 0) {
    cudaGetLastError();
    return 0;
  }
  cached_dev = dev;
  cached = 2 * clusters;
  return cached;
}

bool decode_tc_supported(const DecodeArgs& a) {
  TcParams tp;
  return tc_params(a, tp) && (a.plan.chunk % kTile) == 0;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
  TcParams tp;
  if (!tc_params(a, tp)) return cudaErrorInvalidValue;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  // 5-D view of the cache: [64 elements of a chunk][rows of a run group]
  // [run groups of a block][9 chunks][blocks].  Mode 0: a run group is the
  // D*I rows that hold one run of every shard; mode 1: one group of
  // block_size rows.  The chunk dimension (stride 128 B) comes after the row
  // dimensions, so one box can carry several chunks of the same rows: CTA 0
  // boxes carry chunks 0-3, CTA 1 boxes chunks 4-8 (kind 2: one chunk).
  const int bs = a.block_size;
  const cuuint64_t DI = tp.mode_whole_blocks ? 1 : static_cast<cuuint64_t>(a.D) * a.I;
  const cuuint64_t groups = tp.mode_whole_blocks ? static_cast<cuuint64_t>(bs) : bs / DI;
  const cuuint64_t row = kKDim * 2;
  cuuint64_t dims[5] = {64, DI, groups, 9, static_cast<cuuint64_t>(a.num_blocks)};
  cuuint64_t strides[4] = {row, tp.mode_whole_blocks ? row : row * DI, 128, row * bs};
  cuuint32_t box[5] = {64, static_cast<cuuint32_t>(tp.run), static_cast<cuuint32_t>(tp.box_rows / tp.run), 1, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUtensorMap m0, m1;
  void* base = const_cast<__nv_bfloat16*>(a.kv);
  box[3] = tp.kind == 2 ? 1 : 4;
  if (enc(&m0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  box[3] = tp.kind == 2 ? 1 : 5;
  if (enc(&m1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
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
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel, m0, m1, a, tp);
}

}  // namespace dcp
