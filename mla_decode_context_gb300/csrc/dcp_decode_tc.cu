// Tensor-core split-KV MLA decode for sm_103a (tcgen05 + TMEM + DSMEM).
//
// One work unit = (query row r, shard d, split s): all H <= 128 heads of the
// row (the MMA M dimension) against the split's shard tokens, in tiles of 32
// tokens.  A unit runs on a cluster of two CTAs with different jobs:
//   score CTA (rank 0)  holds Q (128 x 576 bf16 = 288 TMEM columns), computes
//                       S(j) = Q K(j)^T as three thirds over dims [0, 192),
//                       [192, 384), [384, 576) (12 tcgen05.mma each, M=128
//                       N=32 K=16, A from TMEM, issued by three warps into
//                       three accumulators that the softmax adds), runs the
//                       online softmax and
//                       ships P(j) (bf16, 8 KB) plus each head's running max
//                       to the value CTA;
//   value CTA (rank 1)  holds O (128 x 512 fp32 = all 512 TMEM columns),
//                       rescales O when a running max moves, accumulates
//                       O += P(j) V(j) (4 tcgen05.mma, N=256 K=16, both
//                       operands in shared memory) and writes O / l.
// No tensor-core work is duplicated, and the CTAs are coupled one way only
// (P and the max go from score to value), so neither waits on a round trip to
// the other inside the tile loop.
//
// Each tile is read from HBM once, with 16-byte cp.async, one shard token
// per row, straight into the 128B-swizzled chunk-major layout the MMAs read.
// The score CTA's stage ring holds the whole tile for S; the value CTA holds
// V in a 7-slot "own" ring (chunks 4-7) and a 4-slot receive ring (chunks
// 0-3):
//   bf16 cache: each CTA loads what it needs, the second read of a line
//     hitting L2 (DRAM bytes stay 1.01x the tile bytes): the score CTA all
//     nine chunks (36 KB), the value CTA chunks 4-7 with its producers and
//     chunks 0-3 with its warps 19-22 (idle otherwise).  Only P crosses the
//     cluster, so neither CTA's ring waits on the other's loads;
//   fp8 cache: the codes are widened once, by the CTA that loads them: the
//     score CTA loads chunks 0-3 and 8, the value CTA chunks 4-7, and each
//     forwards the widened 16 KB its peer lacks with one DSMEM bulk copy.
// A DSMEM copy was measured at ~900 cycles of round trip plus ~47 cycles per
// KB, so each direction carries at most 24 KB per tile.
//
// While an SM streams cp.async, its shared-memory loads, proxy fences and
// st.async take ~500 cycles each and a release-ordered remote arrival
// thousands, whereas mbarrier waits, local arrivals, bulk copies and tcgen05
// operations stay at tens of cycles (measured on GB300).  So every per-tile
// loop below is built from the cheap kind: one warp fences a ring slot and
// arrives on the barrier its consumers wait on, the slot-consumed signal
// across the cluster is a relaxed arrival, P and the running max travel by
// bulk copy, and the softmax groups share their maxima without waiting.
// Row-by-row addressing takes any paging geometry (block size, shard count,
// interleave); rows that must not be read (past the split, bad block ids)
// are zero-filled.  (TMA boxes were measured to cost a few hundred cycles
// of issue each, and the shard-strided rows of small interleaves allow only
// 8-row boxes, which capped the stream well below HBM bandwidth.  One SM's
// cp.async stream could carry whole rows, but the score CTA loading every
// chunk itself measured no faster on long contexts and slower on batched
// ones, hence the split.)
//
// Warp roles (736 threads):
//   warps 0-3   score: Q load, then softmax group 0 (thread = head = TMEM
//                      lane; even tiles)
//               value: max tracking and O rescale; epilogue columns 0-255
//   warps 4-9   score: (4-7 also Q load) S issuers: warp 4 + 3i + k issues
//                      third k of S for tiles j = i mod 2 into S slot i (a
//                      tcgen05.mma holds its issuing thread far longer than
//                      an N=32 product takes, so issue is spread over warps)
//               value: 4-7 epilogue columns 256-511; 8 forwarder (fp8:
//                      own ring -> score stage); 9 receive-ring arrivals and
//                      the own slot's proxy fence for PV
//   warp 10     both:  TMEM allocation; score: proxy fence of the stage's
//                      own rows, forwarder (fp8: stage -> receive ring);
//                      value: PV issuer
//   warps 11-18 both:  producers (cp.async; the score CTA's wait until Q has
//                      left stages 0-3 for TMEM)
//   warps 19-22 score: softmax group 1 (odd tiles)
//               value: bf16 cache: receive-ring producers (chunks 0-3 of
//                      every tile)
// Every wait is bounded (a timeout sets DCP_DEVERR_TIMEOUT and ends the unit).
#include "dcp_kernels.h"
#include "dcp_sm100.cuh"

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <cstring>
#include <mutex>

namespace dcp {
namespace {

using namespace sm100;

constexpr int kTile = 32;                        // tokens per tile (MMA N of S, K of PV)
constexpr int kStages = 5;                       // score CTA: stage ring
constexpr int kNch = 9;                          // 64-dim chunks of a latent row
constexpr int kChunkBytes = kTile * 128;         // 32 rows x 64 bf16, 128B-swizzled
constexpr int kStageBytes = kNch * kChunkBytes;  // 36 KB
constexpr int kProdWarp0 = 11, kProdWarps = 8;   // producer warps: two groups of 4 (alternate tiles)
constexpr int kGroupThreads = 32 * kProdWarps / 2;
constexpr int kHalfBytes = 4 * kChunkBytes;      // 4 chunks: forwarded each way per tile
constexpr int kOwn = 7;                          // value CTA: own ring slots (chunks 4-7)
constexpr int kRecv = 4;                         // value CTA: receive ring slots (chunks 0-3)
constexpr int kSBuf = 2;                         // S slots (three 32-column thirds each) in TMEM
constexpr int kSParts = 3;                       // K-parts of S, one issuing warp each
constexpr int kPSlots = 4;                       // P slots in the value CTA
constexpr int kPBytes = 128 * kTile * 2;         // P tile: 128 rows x 32 bf16, 64B-swizzled
constexpr int kPWarpBytes = kPBytes / 4;         // one softmax warp's 32 rows
constexpr int kPSlotBytes = 9216;                // P tile + running max per head (+ pad)
constexpr uint32_t kPTx = kPBytes + 128 * 4;     // bytes that fill one P slot
constexpr int kSmWarp1 = kProdWarp0 + kProdWarps;  // score: second softmax group (4 warps)
constexpr int kThreads = 32 * (kSmWarp1 + 4);
constexpr float kRescaleLog2 = 8.0f;

// TMEM columns
constexpr uint32_t kColQ = 0;    // score: 288 columns of Q, 2 bf16 per column
constexpr uint32_t kColS = 288;  // score: 2 slots x 3 thirds x 32 columns of S
constexpr uint32_t kColO = 0;    // value: 512 columns of O
constexpr uint32_t kTmemCols = 512;

struct __align__(8) Bars {
  uint64_t kv_loaded[kStages];  // score: own rows of tile j landed (every thread of tile j's producer group)
  // kv_full (score): the whole tile j is in its stage for S: (fp8) the value
  // CTA's 16 KB landed (armed by a producer), the four producer warps of the
  // tile wrote their bytes of its row mask, and the forwarder has made this
  // CTA's own rows visible to the tensor cores
  uint64_t kv_full[kStages];
  // s_done (both CTAs): the score CTA's stage of tile j is free again: all
  // three parts of S(j) done (fp8: and chunks 0-3 of tile j have landed in
  // the value CTA)
  uint64_t s_done[kStages];
  uint64_t own_loaded[kOwn];    // value: rows of tile j in own slot j % kOwn (every thread of its producer group)
  uint64_t own_free[kOwn];      // value: PV(j) done with own slot j % kOwn
  // value: chunks 0-3 of tile j landed in receive slot j % kRecv (bf16: every
  // thread of the receive-ring producers; fp8: the score CTA's copy)
  uint64_t v_full[kRecv];
  // both (multicast commit of PV(j)): receive slot j % kRecv may refill
  // (bf16: the value CTA's receive-ring producers wait; fp8: the score CTA's
  // forwarder)
  uint64_t v_free[kRecv];
  uint64_t s_full[kSBuf];     // score: the three parts' commits + part 0's arrival
  uint64_t s_free[kSBuf];     // score: the softmax has read the slot (4 warps)
  uint64_t q_staged;          // score: Q is in shared memory (threads of warps 0-7)
  uint64_t q_ready;           // score: Q is in TMEM and stages 0-3 are free again (warps 0-7)
  uint64_t q_gone;            // value (fp8): the score CTA's stages no longer hold Q (remote arrival)
  uint64_t p_full[kPSlots];   // value: P(j) and the max of tile j arrived
  uint64_t p_free[kPSlots];   // both (multicast commit of PV(j)); the score CTA waits on it
  // p_ok (value): PV(j) may go: the max is checked and O rescaled if needed
  // (4 warps), and both halves of V(j) are visible to the tensor cores (the
  // receive-ring warp)
  uint64_t p_ok[kPSlots];
  uint64_t pv_done[kPSlots];  // value: PV(j) completes phase j / kPSlots of pv_done[j % kPSlots]
  uint64_t o_final;           // value: last PV complete
  uint64_t fin_l;             // value: 1/l of every head arrived from the score CTA
  uint64_t fin[1 + kSParts * kSBuf];  // each issuing warp's MMAs complete
  uint64_t m_pub[8];          // score: running max after tile j posted (phase j / 8 of m_pub[j % 8]; 4 warps)
  // score: how many of its tiles producer group g has claimed a stage for
  // (written by the group's first warp, read by the other group)
  int32_t claimed[2];
  uint64_t sm_fin;            // score: both softmax groups' final l and m written (8 warps)
  uint64_t never;             // test hook only: initialised, never arrived on
  // score: valid rows of tile j in mask[j % 16] (written by the producer
  // before it arms kv_full; the slot is rewritten 16 tiles later, long after
  // the softmax of tile j has read it: a producer nine or more tiles ahead
  // needs PV(j), hence P(j), done)
  uint32_t mask[16];
  uint32_t tmem;
  int32_t abort;
};

constexpr int kOffStages = 0;                            // score: stage ring
constexpr int kOffOwn = 0;                               // value: own ring
constexpr int kOffRecv = kOwn * kHalfBytes;              // value: receive ring
constexpr int kOffP = kStages * kStageBytes;             // value: P slots; score: P staging
constexpr int kOffFin = kOffP + kPSlots * kPSlotBytes;   // value: 1/l per head
constexpr int kOffSm = kOffFin + 512;                    // score: running max per tile (8 x 128), final l, m
constexpr int kOffBars = kOffSm + 12 * 128 * 4;
constexpr int kSmemBytes = kOffBars + static_cast<int>(sizeof(Bars)) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory per CTA");

// Score CTA stage ring: chunk c of stage st (32 rows x 128 B, 128B-swizzled).
__host__ __device__ constexpr int stage_chunk_off(int st, int c) { return kOffStages + st * kStageBytes + c * kChunkBytes; }
static_assert(kPSlotBytes % 1024 == 0 && kOffP % 1024 == 0, "P tiles must sit on swizzle-atom boundaries");
static_assert(kOffRecv + kRecv * kHalfBytes <= kOffP, "value CTA rings overlap the P slots");
// The receive warp's p_ok arrival for tile j + kPSlots must not land in tile
// j's phase: it waits for chunks 0-3 of that tile, whose receive slot is
// refilled only after PV(j + kPSlots - kRecv), which is PV(j) or later only
// when kRecv <= kPSlots.
static_assert(kRecv <= kPSlots, "a receive ring deeper than the P slots lets p_ok phases mix tiles");

// Cycle accounting for performance work, compiled only with -DDCP_TRACE=R
// (never in the library build): the warps of role R (1 producers, 2 score
// forwarder, 3 S issuers, 4 softmax, 6 value forwarder, 7 receive warp, 8 PV
// issuer, 9 value max / epilogue warps) add clock64 deltas into eight
// counters (TR_LAP(R, k): time since the last mark goes to counter k), and
// lane 0 of every warp of the first kTraceClusters clusters stores them at
// the end, counter 7 being the warp's whole life.  One role per build keeps
// the counters out of the other roles' registers.  Every CTA also records
// its SM and the global timer at entry and at exit.
#ifdef DCP_TRACE
constexpr int kTraceClusters = 16;
constexpr int kTraceCtas = 1024;
__device__ __align__(16) uint32_t g_dcp_trace[kTraceClusters * 2][32][8];
__device__ __align__(16) unsigned long long g_dcp_timeline[kTraceCtas][8];  // t_entry, t_exit, smid, unit, clk_entry, clk_exit, t_init
__device__ __forceinline__ unsigned long long tr_globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define TR_ENTRY()                                                                      \
  const unsigned long long tr_entry = threadIdx.x == 0 ? tr_globaltimer() : 0ull;       \
  const unsigned long long tr_clk_entry = threadIdx.x == 0 ? clock64() : 0ull
#define TR_INIT()                                                     \
  if (threadIdx.x == 0 && blockIdx.x < kTraceCtas) g_dcp_timeline[blockIdx.x][6] = tr_globaltimer(); \
  uint32_t tr_c[8] = {0, 0, 0, 0, 0, 0, 0, 0};                       \
  const uint32_t tr_start = static_cast<uint32_t>(clock64());         \
  uint32_t tr_t = tr_start
#define TR_MARK(r)                                                    \
  do {                                                                \
    if ((r) == DCP_TRACE) tr_t = static_cast<uint32_t>(clock64());    \
  } while (0)
#define TR_LAP(r, k)                                                  \
  do {                                                                \
    if ((r) == DCP_TRACE) {                                           \
      const uint32_t tr_n = static_cast<uint32_t>(clock64());         \
      tr_c[k] += tr_n - tr_t;                                         \
      tr_t = tr_n;                                                    \
    }                                                                 \
  } while (0)
#define TR_DUMP()                                                                               \
  do {                                                                                          \
    if (blockIdx.x < 2 * kTraceClusters && (threadIdx.x & 31) == 0) {                           \
      tr_c[7] = static_cast<uint32_t>(clock64()) - tr_start;                                    \
      uint4* tr_d = reinterpret_cast<uint4*>(&g_dcp_trace[blockIdx.x][threadIdx.x >> 5][0]);     \
      tr_d[0] = make_uint4(tr_c[0], tr_c[1], tr_c[2], tr_c[3]);                                 \
      tr_d[1] = make_uint4(tr_c[4], tr_c[5], tr_c[6], tr_c[7]);                                 \
    }                                                                                           \
  } while (0)
#define TR_EXIT(unit)                                                                           \
  do {                                                                                          \
    if (threadIdx.x == 0 && blockIdx.x < kTraceCtas) {                                          \
      uint32_t smid;                                                                            \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));                                         \
      g_dcp_timeline[blockIdx.x][0] = tr_entry;                                                 \
      g_dcp_timeline[blockIdx.x][1] = tr_globaltimer();                                         \
      g_dcp_timeline[blockIdx.x][2] = smid;                                                     \
      g_dcp_timeline[blockIdx.x][3] = static_cast<unsigned long long>(unit);                    \
      g_dcp_timeline[blockIdx.x][4] = tr_clk_entry;                                             \
      g_dcp_timeline[blockIdx.x][5] = clock64();                                                \
    }                                                                                           \
  } while (0)
#else
#define TR_ENTRY() do {} while (0)
#define TR_INIT() do {} while (0)
#define TR_MARK(r) do {} while (0)
#define TR_LAP(r, k) do {} while (0)
#define TR_DUMP() do {} while (0)
#define TR_EXIT(unit) do {} while (0)
#endif

__device__ __forceinline__ void report(int32_t* dev_error, uint32_t bits) {
  if (dev_error) atomicOr(dev_error, static_cast<int32_t>(bits));
}

__device__ __forceinline__ bool aborted(Bars& bar) { return *reinterpret_cast<volatile int32_t*>(&bar.abort) != 0; }

__device__ __forceinline__ void set_abort(Bars& bar, int32_t* dev_error) {
  report(dev_error, DCP_DEVERR_TIMEOUT);
  atomicExch(&bar.abort, 1);
}

// Two FP8 E4M3 codes -> bf16x2 of code x s.  Exact: E4M3 values convert
// exactly to half and to fp32, s is a power of two, and a code has at most 4
// significant bits, so the product (in fp32 range) is exact in bf16 too.
// (s2: the scale in both halves of a packed fp32 pair; one f32x2 multiply.)
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t codes, uint64_t s2) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes & 0xffffu), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  float lo, hi;
  f2_unpack(f2_mul(f2_pack(f.x, f.y), s2), lo, hi);
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// kFp8: the cache holds FP8 E4M3 codes (576 bytes a row) with one fp32 scale
// per slot; the producers widen them to bf16 on their way into shared
// memory, so everything downstream is the same as for a bf16 cache.
template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(DecodeArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  TR_ENTRY();
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  Bars& bar = *reinterpret_cast<Bars*>(smem + kOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();
  const bool score = cta == 0;
  const uint32_t peer = cta ^ 1u;

  const int64_t unit = a.unit_order ? __ldg(a.unit_order + (blockIdx.x >> 1)) : (blockIdx.x >> 1);
  const UnitCoords uc = unit_coords(a, unit);
  const int r = uc.r;
  const int d = a.d0 + uc.dd;  // shard (of D)
  const int s = uc.s;

  if (score && warp < 8) {
    // Q load, issued first (it depends only on the row) so that its latency
    // overlaps the row lookup's loads and the set-up.  The 147 KB of Q (128
    // heads x 576 dims, the same for every unit of a row) come in with one
    // round of cp.async into stages 0-3 (unused until Q is in TMEM): head h
    // at 1152 h, its 16-byte unit u at position u ^ (h & 7) within each
    // 8-unit group.  Heads h >= H are zero.
    const unsigned char* qb = reinterpret_cast<const unsigned char*>(a.q + static_cast<int64_t>(r) * a.q_stride_tok);
    const uint32_t qs = smem_u32(smem) + kOffStages;
    for (int p = threadIdx.x; p < 128 * 72; p += 256) {
      const int hh = p / 72, u = p - hh * 72;
      const int us = (u & ~7) | ((u & 7) ^ (hh & 7));
      cp_async16_zfill(qs + hh * 1152 + us * 16, qb + (hh < a.H ? hh : 0) * 1152 + u * 16, hh < a.H ? 16u : 0u);
    }
    cp_async_commit();
  }

  const RowInfo ri = resolve_row(a.seq_lens, a.qsl, a.B, r, a.max_seq_len, a.max_q_len);
  if (ri.err && threadIdx.x == 0 && cta == 0 && d == a.d0 && s == 0) report(a.dev_error, ri.err);
  const int32_t n_local = ri.padding ? 0 : local_len(ri.L, d, a.D, a.I);
  const int32_t lo = s * a.plan.chunk;
  const int32_t hi = min(n_local, lo + a.plan.chunk);
  const int ntiles = lo < hi ? (hi - lo + kTile - 1) / kTile : 0;
  const int64_t pair0 = ((static_cast<int64_t>(s) * a.Dn + (d - a.d0)) * a.T + r) * a.H;

  if (ntiles == 0) {
    if (score && warp < 8) cp_async_wait<0>();  // the Q copies land before the CTA leaves
    // empty shard / split or padding row: masked at the source, no KV read
    if (warp < 4) {
      const int h = threadIdx.x;
      if (h < a.H) {
        if (score) {
          a.lse_dst[pair0 + h] = -INFINITY;
        } else {
          // a zero output row: 2 KB in fp32, 1 KB in bf16
          const int64_t row_bytes = a.o_bf16 ? 2 * kLatent : 4 * kLatent;
          uint4* o = reinterpret_cast<uint4*>(static_cast<unsigned char*>(a.O_dst) + (pair0 + h) * row_bytes);
          for (int i = 0; i < row_bytes / 16; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    TR_EXIT(unit);
    return;
  }


  // ---------------------------------------------------------------- setup
  // (by a thread of a warp that issued no Q copies, so that the barrier
  // stores do not queue behind its own)
  if (threadIdx.x == 32 * kProdWarp0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar.kv_loaded[i], kGroupThreads);
      mbar_init(&bar.kv_full[i], 5);  // 4 producer warps of the tile's group + the forwarder
      mbar_init(&bar.s_done[i], kFp8 ? kSParts + 1 : kSParts);
    }
    for (int i = 0; i < kOwn; ++i) { mbar_init(&bar.own_loaded[i], kGroupThreads); mbar_init(&bar.own_free[i], 1); }
    for (int i = 0; i < kRecv; ++i) { mbar_init(&bar.v_full[i], kFp8 ? 1 : kGroupThreads); mbar_init(&bar.v_free[i], 1); }
    for (int i = 0; i < kSBuf; ++i) { mbar_init(&bar.s_full[i], kSParts + 1); mbar_init(&bar.s_free[i], 4); }
    mbar_init(&bar.q_staged, 256);
    mbar_init(&bar.q_ready, 8);
    mbar_init(&bar.q_gone, 1);
    for (int i = 0; i < kPSlots; ++i) {
      mbar_init(&bar.p_full[i], 1);
      mbar_init(&bar.p_free[i], 1);
      mbar_init(&bar.p_ok[i], 5);
      mbar_init(&bar.pv_done[i], 1);
    }
    mbar_init(&bar.o_final, 1);
    mbar_init(&bar.fin_l, 1);
    for (int i = 0; i < 1 + kSParts * kSBuf; ++i) mbar_init(&bar.fin[i], 1);
    for (int i = 0; i < 8; ++i) mbar_init(&bar.m_pub[i], 4);
    bar.claimed[0] = bar.claimed[1] = 0;
    mbar_init(&bar.sm_fin, 8);
    mbar_init(&bar.never, 1);
    bar.abort = 0;
    fence_mbar_init();
    if (!score) {
      // every P slot starts free: expect the first P tile and max column
      for (int i = 0; i < kPSlots; ++i) mbar_arrive_expect_tx(&bar.p_full[i], kPTx);
      if (kFp8)
        for (int i = 0; i < kRecv; ++i) mbar_arrive_expect_tx(&bar.v_full[i], kHalfBytes);
      mbar_arrive_expect_tx(&bar.fin_l, 128 * 4);
    }
  }
  if (warp == 10) {
    tmem_alloc(&bar.tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // peer's barriers initialised and armed before any remote operation
  tc_fence_after();
  const uint32_t tbase = bar.tmem;
  TR_INIT();
  if (score && warp < 8) {
    // Q -> TMEM, once the copies issued before the set-up have landed:
    // thread = head = lane of the warp's lane quarter moves its row to TMEM
    // (warps 0-3 the even chunks, 4-7 the odd ones): dim k goes to column
    // k / 2 (low half = even k).
    cp_async_wait<0>();
    mbar_arrive(&bar.q_staged);
    const bool staged = __all_sync(0xffffffffu, mbar_wait(&bar.q_staged, 0));
    const int h = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    if (staged) {
      for (int c = warp >> 2; c < kNch; c += 2) {
        uint32_t v[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // unit k of the chunk sits at position k ^ (h & 7)
          const uint4 x = *reinterpret_cast<const uint4*>(smem + kOffStages + h * 1152 + (c * 8 + (k ^ (h & 7))) * 16);
          v[4 * k] = x.x; v[4 * k + 1] = x.y; v[4 * k + 2] = x.z; v[4 * k + 3] = x.w;
        }
        tmem_st32(lane_addr + kColQ + 32 * c, v);
      }
    } else {
      set_abort(bar, a.dev_error);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar.q_ready);
    TR_LAP(4, 6);  // score warps 0-7: Q load
  }

  // the request's table row (global layout) or this shard's row of it (per-shard layout)
  const int32_t* trow = a.block_table + static_cast<int64_t>(ri.b) * a.bt_stride +
                        (a.local_tables ? static_cast<int64_t>(d - a.d0) * a.bt_shard_stride : 0);
  const uint32_t smem_base = smem_u32(smem);
  int pdone = 0;  // value, warps 0-3: P tiles received

  if ((warp >= kProdWarp0 && warp < kSmWarp1) || (!kFp8 && !score && warp >= kSmWarp1)) {
    // ----------------------------------------------------------- producers
    // Two groups of four warps take alternate tiles (a producer thread's
    // issue is latency-bound, so two tiles are in flight at once).  Warp gw
    // of a group owns rows 8 gw .. 8 gw + 7 of the tile, four at a time:
    // eight lanes per row, lane x copying the x-th 16-byte unit of every
    // chunk the CTA loads itself (chunks 0-3 and the rope chunk 8 into the
    // score CTA's stage, chunks 4-7 into the value CTA's own slot, laid out
    // as the stage's chunks are), so each copy instruction reads four whole
    // 128-byte lines.  Each thread resolves its own two rows (shard token ->
    // cache row) one of the group's tiles ahead: no values move between
    // lanes, which keeps the SM's memory-instruction queue, busy with the
    // copies, free of shuffles.  Each thread's copies of a tile arrive on
    // kv_loaded / own_loaded by themselves when they complete; the consumers
    // fence them into the async proxy.
    const int group = (warp - kProdWarp0) >> 2;
    const int gw = (warp - kProdWarp0) & 3;
    const int x = lane & 7;
    const int row0 = 8 * gw + (lane >> 3), row1 = row0 + 4;
    const int nch = score ? (kFp8 ? 5 : 9) : 4;  // chunks this CTA loads itself
    const unsigned char* kvb = reinterpret_cast<const unsigned char*>(a.kv);
    // bf16 cache, value CTA: group 2 (warps 19-22) loads chunks 0-3 of every
    // tile into the receive ring, one tile after another; groups 0 and 1 take
    // alternate tiles' chunks 4-7 as in the score CTA
    const bool vrecv = !kFp8 && !score && group == 2;
    const int step = vrecv ? 1 : 2, j0 = vrecv ? 0 : group;
    uint64_t* own_free = score ? bar.s_done : (vrecv ? bar.v_free : bar.own_free);
    uint64_t* own_loaded = score ? bar.kv_loaded : (vrecv ? bar.v_full : bar.own_loaded);
    const int nslots = score ? kStages : (vrecv ? kRecv : kOwn);
    const int32_t DI = a.D * a.I, dI = d * a.I;
    bool in_n[2] = {false, false};
    int32_t off_n[2] = {0, 0}, blk_n[2] = {-1, -1};  // row within its block, block id
    auto fetch = [&](int jj) {  // positions fit in 32 bits (seq_lens are int32)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int32_t l = lo + jj * kTile + (e ? row1 : row0);
        in_n[e] = l < hi;
        // the table index: the shard token's position, or (per-shard
        // layout) the local token index itself
        const int32_t lq = fast_div(l, a.div_I);
        const int32_t pos = in_n[e] ? (a.local_tables ? l : lq * DI + dI + (l - lq * a.I)) : 0;
        const int32_t pb = fast_div(pos, a.div_bs);
        off_n[e] = pos - pb * a.block_size;
        blk_n[e] = in_n[e] ? __ldg(trow + pb) : -1;
      }
    };
    // rows of the tile whose block ids are in in_n / off_n / blk_n
    auto rows_of = [&](bool (&valid)[2], int32_t (&crow)[2], bool& bad) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        valid[e] = in_n[e] && blk_n[e] >= 0 && blk_n[e] < a.num_blocks;
        // cache row (fits in 31 bits: the library only takes caches of < 2^31 rows)
        crow[e] = valid[e] ? blk_n[e] * a.block_size + off_n[e] : 0;
      }
      bad = (in_n[0] && !valid[0]) || (in_n[1] && !valid[1]);
    };
    // FP8 cache: this thread's codes (8 per row and chunk) and row scales of
    // a tile, loaded one of the group's tiles ahead of their conversion
    uint2 codes[2][5];
    float rscale[2] = {0.f, 0.f};
    auto load_codes = [&](const bool (&valid)[2], const int32_t (&crow)[2]) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const unsigned char* src_row = kvb + static_cast<int64_t>(crow[e]) * kKDim + x * 8;
        rscale[e] = valid[e] ? __ldg(a.kv_scale + crow[e]) : 0.f;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
          const int c = score ? (i < 4 ? i : 8) : 4 + i;
          codes[e][i] = (valid[e] && i < nch) ? __ldg(reinterpret_cast<const uint2*>(src_row + c * 64)) : make_uint2(0u, 0u);
        }
      }
    };
    bool valid_n[2] = {false, false};
    int32_t crow_n[2] = {0, 0};
    bool bad_n = false;
    fetch(j0);
    if constexpr (kFp8) {
      rows_of(valid_n, crow_n, bad_n);
      load_codes(valid_n, crow_n);
      if (group + 2 < ntiles) fetch(group + 2);
    }
    bool ok = true;
    if (score) ok = __all_sync(0xffffffffu, mbar_wait(&bar.q_ready, 0));
    TR_LAP(1, 5);  // producers: waiting for Q to leave the stages
    // slot j % nslots and the parity of j / nslots, kept as running values
    // (nslots is 5 or 7 by CTA, so the compiler cannot fold the division)
    int st = j0, round = 0;
    // the other group's claim count as last read: it only grows, so it is
    // read again only when it falls short of what a tile needs (below)
    int32_t other_claimed = 0;
    for (int j = j0; j < ntiles && ok; j += step) {
      // score CTA: the other group has claimed its stage for tile j - 5,
      // which it did after S(j - 10) finished.  So the stage-free barrier
      // below is at S(j - 5)'s phase or past it, and its parity can only
      // mean S(j - 5), however the copies and MMAs of other tiles complete.
      // (A monotonic count, not a parity wait: the groups may drift apart.
      // Tested first in the iteration, before this tile's global loads are
      // issued, so that the shared-memory read does not queue behind them.)
      if (score && j >= 5) {
        const int32_t need = ((j - 5) >> 1) + 1;
        for (uint32_t i = 0; other_claimed < need && i < kWaitLimit; ++i)
          other_claimed = ld_relaxed_shared(&bar.claimed[group ^ 1]);
        ok = __all_sync(0xffffffffu, other_claimed >= need);
      }
      if (!ok) break;
      bool valid[2];
      int32_t crow[2];
      bool bad;
      uint2 cur[2][5];
      float cur_scale[2];
      if constexpr (kFp8) {
        // this tile's codes were loaded last time round; load the group's
        // next tile's now, and fetch the block ids of the one after
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          valid[e] = valid_n[e];
          crow[e] = crow_n[e];
          cur_scale[e] = rscale[e];
#pragma unroll
          for (int i = 0; i < 5; ++i) cur[e][i] = codes[e][i];
        }
        bad = bad_n;
        if (j + 2 < ntiles) {
          rows_of(valid_n, crow_n, bad_n);
          load_codes(valid_n, crow_n);
          if (j + 4 < ntiles) fetch(j + 4);
        }
      } else {
        rows_of(valid, crow, bad);
        if (j + step < ntiles) fetch(j + step);
      }
      // the abort flag is read here and tested after this tile's copies are
      // issued, so that its shared-memory latency overlaps them
      const bool ab = aborted(bar);
      TR_LAP(1, 2);  // producers: block ids, loop
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&own_free[st], (round & 1) ^ 1));
      TR_LAP(1, 0);  // producers: waiting for a free slot
      if (!ok) break;
      if (score && gw == 0 && lane == 0) st_relaxed_shared(&bar.claimed[group], (j >> 1) + 1);
      if (__any_sync(0xffffffffu, bad) && score && lane == 0) report(a.dev_error, DCP_DEVERR_BAD_BLOCK);
      if (score) {
        // this warp's 8 rows of the tile's mask (lanes 8q .. 8q + 7 hold rows
        // 8 gw + q and 8 gw + 4 + q), then its arrival on kv_full releases
        // that byte to the softmax; warp 0 of the group also arms kv_full for
        // the value CTA's 16 KB (tile j - 5 is done with the stage, so its
        // previous phase is over)
        const unsigned v0 = __ballot_sync(0xffffffffu, valid[0]), v1 = __ballot_sync(0xffffffffu, valid[1]);
        if (lane == 0) {
          uint32_t m8 = 0;
#pragma unroll
          for (int q = 0; q < 4; ++q) m8 |= (((v0 >> (8 * q)) & 1u) << q) | (((v1 >> (8 * q)) & 1u) << (4 + q));
          reinterpret_cast<volatile uint8_t*>(&bar.mask[j & 15])[gw] = static_cast<uint8_t>(m8);
          if (kFp8 && gw == 0) mbar_arrive_expect_tx(&bar.kv_full[st], kHalfBytes);
          else mbar_arrive(&bar.kv_full[st]);
        }
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = e ? row1 : row0;
        const unsigned char* src_row = kvb + static_cast<int64_t>(crow[e]) * (kKDim * 2) + x * 16;
        const uint32_t src_bytes = valid[e] ? 16u : 0u;
        const uint32_t swz = static_cast<uint32_t>(row * 128 + ((x ^ (row & 7)) << 4));
#pragma unroll
        for (int i = 0; i < nch; ++i) {
          // score: chunks 0-8 (fp8: 0-3, 8) at stage_chunk_off(st, c);
          // value: chunks 4-7 at its own slot's chunk offsets 0-3, or
          // (receive-ring producers) chunks 0-3 at the receive slot's
          const int c = score ? (kFp8 ? (i < 4 ? i : 8) : i) : (vrecv ? i : 4 + i);
          const uint32_t dst = score ? smem_base + stage_chunk_off(st, c) + swz
                                     : smem_base + (vrecv ? kOffRecv : kOffOwn) + st * kHalfBytes + i * kChunkBytes + swz;
          if constexpr (kFp8) {
            // 8 codes -> 8 bf16 (zeros for rows that were not loaded)
            const uint2 w = cur[e][i];
            const uint64_t sc = f2_pack(cur_scale[e], cur_scale[e]);
            const uint4 v = make_uint4(e4m3x2_to_bf16x2(w.x, sc), e4m3x2_to_bf16x2(w.x >> 16, sc),
                                       e4m3x2_to_bf16x2(w.y, sc), e4m3x2_to_bf16x2(w.y >> 16, sc));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
          } else {
            cp_async16_zfill(dst, src_row + c * 128, src_bytes);
          }
        }
      }
      // (fp8: this thread's stores are done; the consumers fence them into
      // the async proxy after this arrival, as they do the copies')
      if constexpr (kFp8) mbar_arrive(&own_loaded[st]);
      else cp_async_mbar_arrive_noinc(&own_loaded[st]);
      TR_LAP(1, 1);  // producers: issuing the copies
      if (__any_sync(0xffffffffu, ab)) {
        ok = false;
        break;
      }
      st += step;
      if (st >= nslots) {
        st -= nslots;
        ++round;
      }
    }
    if (!ok) set_abort(bar, a.dev_error);
    cp_async_wait<0>();
  } else if (score && warp == 10) {
    // ------------------------------------------------- score CTA forwarder
    // Two streams of tiles, each in order, served as their conditions come
    // true (non-blocking polls), so that neither waits behind the other:
    //   fence: once this CTA's own rows of tile jf have landed, fence them
    //          into the async proxy and arrive on kv_full (for S);
    //   copy:  (fp8) once tile jc < jf is fenced and the value CTA's receive
    //          slot is free, copy chunks 0-3 (16 KB) into it.  (bf16: the
    //          value CTA loads them itself; jc follows jf.)
    // (kv_loaded(jf + 5) needs S(jf), hence the fence of jf: no parity
    // aliasing.)  The loop gives up after kWaitLimit polls without progress.
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bar.q_ready, 0));
    // fp8: the value CTA's forwards into the stages (which held Q) may start
    if (kFp8 && ok && lane == 0) mbar_arrive_remote(map_peer(smem_u32(&bar.q_gone), peer));
    int jf = 0, jc = 0;
    uint32_t idle = 0;
    while (ok && jc < ntiles) {
      bool moved = false;
      if (jf < ntiles && __all_sync(0xffffffffu, mbar_peek(&bar.kv_loaded[jf % kStages], (jf / kStages) & 1))) {
        fence_proxy_async_smem();  // the producers' cp.async writes -> S and the bulk copy
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.kv_full[jf % kStages]);
        ++jf;
        moved = true;
      }
      if (!kFp8) jc = jf;
      if (kFp8 && jc < jf && __all_sync(0xffffffffu, mbar_peek_cluster(&bar.v_free[jc % kRecv], ((jc / kRecv) & 1) ^ 1))) {
        const int st = jc % kStages, rs = jc % kRecv;
        if (lane == 0)  // chunks 0-3 of the stage -> the receive slot
          bulk_copy_to_peer(map_peer(smem_base + kOffRecv + rs * kHalfBytes, peer), smem + stage_chunk_off(st, 0),
                            kHalfBytes, map_peer(smem_u32(&bar.v_full[rs]), peer));
        __syncwarp();
        ++jc;
        moved = true;
      }
      idle = moved ? 0u : idle + 1u;
      if (moved) TR_LAP(2, 1); else TR_LAP(2, 0);  // forwarder: working / polling
      if (idle > kWaitLimit) ok = false;
    }
    if (!ok) set_abort(bar, a.dev_error);
  } else if (!score && warp == 8) {
    // ------------------------------------------------- value CTA forwarder
    // fp8: own slot j % kOwn (chunks 4-7) -> the score CTA's stage of tile j,
    // once that stage is free (tile j - 5 done there) and no longer holds Q.
    // (bf16: the score CTA loads those chunks itself.)
    bool ok = !kFp8 || __all_sync(0xffffffffu, mbar_wait_cluster(&bar.q_gone, 0));
    TR_LAP(6, 5);
    for (int j = 0; kFp8 && j < ntiles && ok; ++j) {
      const int st = j % kStages, os = j % kOwn;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.own_loaded[os], (j / kOwn) & 1));
      TR_LAP(6, 0);  // value forwarder: waiting for own rows
      ok = ok && __all_sync(0xffffffffu, mbar_wait_cluster(&bar.s_done[st], ((j / kStages) & 1) ^ 1));
      TR_LAP(6, 1);  // value forwarder: waiting for the score stage to be free
      if (!ok) break;
      fence_proxy_async_smem();  // the producers' cp.async writes -> the bulk copy
      if (lane == 0)  // own chunks 4-7 -> chunks 4-7 of the score CTA's stage
        bulk_copy_to_peer(map_peer(smem_base + stage_chunk_off(st, 4), peer), smem + kOffOwn + os * kHalfBytes,
                          kHalfBytes, map_peer(smem_u32(&bar.kv_full[st]), peer));
      __syncwarp();
      TR_LAP(6, 2);  // value forwarder: fence + copy
    }
    if (!ok) set_abort(bar, a.dev_error);
  } else if (!score && warp == 9) {
    // ------------------------------------------------- receive-ring arrivals
    // When tile j's chunks 0-3 land (fp8: copied in), re-arm the slot for
    // tile j + kRecv (that fill needs PV(j) first, so it cannot complete
    // before this) and tell both CTAs that the score CTA's stage of tile j
    // has been read (a relaxed arrival: the copy's reads are complete, and
    // nothing written here needs publishing).  Then, once this CTA's own
    // rows of tile j have landed, fence them (bf16: and the receive slot's
    // rows) into the async proxy and let PV(j) go.  (This warp's arrival
    // for tile j + kPSlots needs v_full(j + kPSlots), hence PV(j) done, so it
    // cannot land in tile j's phase of p_ok.)
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int st = j % kStages, vs = j % kRecv, os = j % kOwn;
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(&bar.v_full[vs], (j / kRecv) & 1));
      TR_LAP(7, 0);  // receive warp: waiting for chunks 0-3
      if (!ok) break;
      if (kFp8 && lane == 0) {
        mbar_arrive_expect_tx(&bar.v_full[vs], kHalfBytes);
        mbar_arrive(&bar.s_done[st]);
        mbar_arrive_remote_relaxed(map_peer(smem_u32(&bar.s_done[st]), peer));
      }
      TR_LAP(7, 1);
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.own_loaded[os], (j / kOwn) & 1));
      TR_LAP(7, 2);  // receive warp: waiting for own rows
      if (!ok) break;
      fence_proxy_async_smem();  // the own (bf16: and receive) slot's cp.async rows -> PV
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.p_ok[j % kPSlots]);
      TR_LAP(7, 3);  // receive warp: fence
    }
    if (!ok) set_abort(bar, a.dev_error);
  } else if (score && warp >= 4 && warp < 10) {
    // ------------------------------------------------------- S MMA issuers
    // warp 4 + 3b + part owns third `part` of S slot b (dims [192 part,
    // 192 part + 192): 12 k-steps) for tiles j = b (mod 2).  Stage layout:
    // chunk-major, 4 KB per 64-dim chunk, 8-row groups 1 KB apart.
    const int b = (warp - 4) / kSParts, part = (warp - 4) % kSParts;
    const uint32_t id_s = idesc_bf16(128, kTile, 0, 0);
    const uint64_t dk = smem_desc(smem_base + kOffStages, 16, 1024, kSwizzle128B);
    const uint32_t dS = tbase + kColS + 96 * b + 32 * part;
    // The part's first k-step: Q columns and the stage's chunk offset.  A
    // tcgen05.mma holds its issuing thread for tens of cycles, and any
    // arithmetic that the next one's operands wait for adds to that, so the
    // operands of a chunk's four MMAs are its base plus constants.
    const uint32_t qa = tbase + kColQ + 96 * part;
    const uint64_t dkp = dk + static_cast<uint64_t>((3 * part * kChunkBytes) >> 4);
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bar.q_ready, 0));
    tc_fence_after();
    TR_LAP(3, 5);
    for (int j = b; ok && j < ntiles; j += kSBuf) {
      const int st = j % kStages, u = j / kSBuf;
      // s_free first: once the softmax has read S(j - 2) it has read every
      // earlier tile, so the stage's previous fill (tile j - 5) is consumed
      // and the kv_full parity below can only mean tile j.  kv_full covers
      // both halves of the tile, this CTA's already fenced into the async
      // proxy by the forwarder.
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_free[b], (u & 1) ^ 1));
      TR_LAP(3, 0);  // S issuer: waiting for the softmax to read the slot
      ok = ok && __all_sync(0xffffffffu, mbar_wait_cluster(&bar.kv_full[st], (j / kStages) & 1));
      TR_LAP(3, 1);  // S issuer: waiting for the tile
      if (!ok) break;
      // rows that were not loaded are zero and only reach S columns the
      // softmax masks.  Part 0's arrival passes on (release after the
      // acquire of kv_full) the producer's write of the tile's mask, which
      // the softmax reads after s_full.
      if (part == 0 && lane == 0) mbar_arrive(&bar.s_full[b]);
      tc_fence_after();
      if (lane == 0) {
        uint64_t bc = dkp + static_cast<uint64_t>((st * kStageBytes) >> 4);
        uint32_t ac = qa;
#pragma unroll 1
        for (int c = 0; c < 3; ++c, bc += kChunkBytes >> 4, ac += 32) {
#pragma unroll
          for (int i = 0; i < 4; ++i) mma_ts(dS, ac + 8 * i, bc + 2 * i, id_s, (c | i) != 0);
        }
        TR_LAP(3, 3);  // S issuer: the 12 MMAs
        mma_commit(&bar.s_full[b]);
        mma_commit_mc(&bar.s_done[st], 0x3);
      }
      __syncwarp();
      TR_LAP(3, 2);  // S issuer: issuing
    }
    if (!ok) set_abort(bar, a.dev_error);
    if (lane == 0) mma_commit(&bar.fin[1 + kSParts * b + part]);
    __syncwarp();
    mbar_wait(&bar.fin[1 + kSParts * b + part], 0);
  } else if (score && (warp < 4 || warp >= kSmWarp1)) {
    // ------------------------------------------------------------- softmax
    // Two groups of four warps take alternate tiles.  Each group keeps its
    // own running max m and the normaliser of its own tiles in that max's
    // scale.  After each tile a group posts its m (m_ring, m_pub), and before
    // tile j it adopts, if larger, the other group's m after tile j - 3 (after
    // tile 0 for tile 1): a lag at which the post is nearly always there
    // already, so neither group waits on the other, and a fixed one, so the
    // result does not depend on timing.  P(j) goes out with the m it was
    // computed with; the value CTA rescales O whenever consecutive tiles' m
    // differ, which happens only around the rare growth of the max (lazy by
    // 2^8).  At the end the two normalisers are brought to the scale of O,
    // which is the m of the last tile that had one.
    const int sg = warp < 4 ? 0 : 1, q4 = warp & 3;
    const int h = q4 * 32 + lane;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(q4 * 32) << 16);
    float* m_ring = reinterpret_cast<float*>(smem + kOffSm);  // [tile % 8][128]: running max after the tile
    float* fin_sh = m_ring + 8 * 128;                         // [group][l, m][128]
    const float sl2 = a.scale * kLog2e;
    float m_used = -INFINITY, l_sum = 0.f;
    const int sw = (h >> 1) & 3;  // 64-byte swizzle of row h
    const uint32_t p_row = static_cast<uint32_t>((h >> 3) * 512 + (h & 7) * 64);
    bool ok = true;
    // failure-path test hook: a wait that runs out (nothing completes `never`)
    if (a.stall_test && sg == 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar.never, 0));
    for (int j = sg; ok && j < ntiles; j += 2) {
      const int b = j % kSBuf, slot = j % kPSlots;
      // the other group's m after tile k, read early so that the load's
      // latency overlaps the wait for S.  Its ring slot takes tile k + 8's
      // max only after the writer has waited for this group's post of tile
      // k + 5, which this group makes after this read.
      float m_other = -INFINITY;
      const int k = j == 1 ? 0 : j - 3;
      if (k >= 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar.m_pub[k & 7], (k >> 3) & 1));
        if (!ok) break;
        m_other = *reinterpret_cast<volatile float*>(&m_ring[(k & 7) * 128 + h]);
      }
      TR_LAP(4, 0);  // softmax: the other group's max
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full[b], (j / kSBuf) & 1));
      TR_LAP(4, 1);  // softmax: waiting for S
      if (!ok) break;
      tc_fence_after();
      const uint32_t mask = *reinterpret_cast<volatile uint32_t*>(&bar.mask[j & 15]);
      uint32_t sr[32], sr2[32];
      tmem_ld32(lane_addr + kColS + 96 * b, sr);
      tmem_ld32(lane_addr + kColS + 96 * b + 32, sr2);
      tmem_wait_ld();
      float sc[32];
#pragma unroll
      for (int i = 0; i < 16; ++i)  // the K-parts of S, pairwise
        f2_unpack(f2_add(f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])),
                         f2_pack(__uint_as_float(sr2[2 * i]), __uint_as_float(sr2[2 * i + 1]))),
                  sc[2 * i], sc[2 * i + 1]);
      tmem_ld32(lane_addr + kColS + 96 * b + 64, sr);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.s_free[b]);
      TR_LAP(4, 2);  // softmax: reading S
#pragma unroll
      for (int i = 0; i < 16; ++i)
        f2_unpack(f2_add(f2_pack(sc[2 * i], sc[2 * i + 1]),
                         f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]))),
                  sc[2 * i], sc[2 * i + 1]);
      // online softmax in base 2: x = s * scale * log2(e), scaled before the
      // mask and the max so that any finite scale (zero and negative too)
      // keeps masked tokens at -inf; masked tokens get weight 0 by selection
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
      for (int i = 0; i < 16; ++i) f2_unpack(f2_mul(f2_pack(sc[2 * i], sc[2 * i + 1]), sl2x2), sc[2 * i], sc[2 * i + 1]);
      if (mask != 0xffffffffu) {
#pragma unroll
        for (int i = 0; i < 32; ++i) sc[i] = (mask >> i) & 1u ? sc[i] : -INFINITY;
      }
      // row max, as a tree
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = fmaxf(fmaxf(sc[4 * i], sc[4 * i + 1]), fmaxf(sc[4 * i + 2], sc[4 * i + 3]));
      const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // adopt the other group's max if it is larger (it only grows)
      if (m_other > m_used) {
        if (m_used != -INFINITY) l_sum *= ex2_approx(m_used - m_other);
        m_used = m_other;
      }
      // lazy rescale: the running max only moves when it would grow by more
      // than 2^8 (the value CTA rescales O by the same factor)
      const bool grow = m_used == -INFINITY ? (tmax != -INFINITY) : (tmax > m_used + kRescaleLog2);
      if (grow) {
        if (m_used != -INFINITY) l_sum *= ex2_approx(m_used - tmax);
        m_used = tmax;
      }
      // (tile j - 8's max, in this slot, was read at tile j - 5, before the
      // other group posted tile j - 3's max, which this group waited for)
      m_ring[(j & 7) * 128 + h] = m_used;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.m_pub[j & 7]);
      // p = 2^(x - m); masked (-inf) scores give exactly 0, and nothing is
      // live while m is still -inf
      const float nm = m_used == -INFINITY ? 0.f : -m_used;
      const uint64_t nmx2 = f2_pack(nm, nm);
      uint32_t pk[16];
      uint64_t ps[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float e0, e1;
        f2_unpack(f2_add(f2_pack(sc[2 * i], sc[2 * i + 1]), nmx2), e0, e1);
        const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
        __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);  // P feeds the PV MMA in bf16
        ps[i & 1] = f2_add(ps[i & 1], f2_pack(p0, p1));     // l (hence the LSE) stays fp32
        pk[i] = *reinterpret_cast<uint32_t*>(&pb);
      }
      float q0, q1, q2, q3;
      f2_unpack(ps[0], q0, q1);
      f2_unpack(ps[1], q2, q3);
      l_sum += (q0 + q1) + (q2 + q3);
      // the slot (and this CTA's staging copy of it) is free once PV(j - kPSlots) is done
      TR_LAP(4, 3);  // softmax: arithmetic
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(&bar.p_free[slot], ((j / kPSlots) & 1) ^ 1));
      TR_LAP(4, 4);  // softmax: waiting for a free P slot
      if (!ok) break;
      unsigned char* stg = smem + kOffP + slot * kPSlotBytes;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(stg + p_row + ((c ^ sw) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      *reinterpret_cast<float*>(stg + kPBytes + 4 * h) = m_used;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        // this warp's 32 rows of P, then its 32 maxima: two bulk copies
        const uint32_t peer_slot = map_peer(smem_base + kOffP + slot * kPSlotBytes, peer);
        const uint32_t peer_full = map_peer(smem_u32(&bar.p_full[slot]), peer);
        bulk_copy_to_peer(peer_slot + q4 * kPWarpBytes, stg + q4 * kPWarpBytes, kPWarpBytes, peer_full);
        bulk_copy_to_peer(peer_slot + kPBytes + q4 * 128, stg + kPBytes + q4 * 128, 128, peer_full);
      }
      TR_LAP(4, 5);  // softmax: P out
    }
    // both groups' normalisers meet here; group 0 finishes the unit
    fin_sh[(2 * sg) * 128 + h] = l_sum;
    fin_sh[(2 * sg + 1) * 128 + h] = m_used;
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar.sm_fin);
    if (!ok) {
      set_abort(bar, a.dev_error);
    } else if (sg == 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.sm_fin, 0)) && !__any_sync(0xffffffffu, aborted(bar));
      if (!ok) {
        set_abort(bar, a.dev_error);
      } else {
        const float l1 = *reinterpret_cast<volatile float*>(&fin_sh[2 * 128 + h]);
        const float m1 = *reinterpret_cast<volatile float*>(&fin_sh[3 * 128 + h]);
        // O is in the scale of the m sent with the last tile that had one
        // (a group's m is final after its last tile and never returns to
        // -inf): the group of tile ntiles - 1, else the other group
        const bool last0 = ((ntiles - 1) & 1) == 0;
        float mo = last0 ? m_used : m1;
        if (mo == -INFINITY) mo = last0 ? m1 : m_used;
        float l = 0.f;
        if (m_used != -INFINITY) l += l_sum * ex2_approx(m_used - mo);
        if (m1 != -INFINITY) l += l1 * ex2_approx(m1 - mo);
        const bool live = l > 0.f;
        st_async_peer_b32(map_peer(smem_base + kOffFin + 4 * h, peer), __float_as_uint(live ? 1.f / l : 0.f),
                          map_peer(smem_u32(&bar.fin_l), peer));
        if (h < a.H) a.lse_dst[pair0 + h] = live ? (mo + log2f(l)) * kLn2 : -INFINITY;
      }
    }
  } else if (!score && warp == 10) {
    // -------------------------------------------------------- PV MMA issuer
    // O accumulates across tiles, so PV(j) is issued in order by one thread.
    // P (K-major, 64-byte swizzle) and V (value dims 0-255 from the receive
    // slot, 256-511 from the own slot, each read MN-major: N atoms = 4 KB
    // chunks, K = tokens in 8-row groups 1 KB apart) both come from shared
    // memory.  Rows that were not loaded are zero, so P = 0 never meets a
    // NaN/Inf value.
    const uint32_t id_o = idesc_bf16(128, 256, 0, 1);
    const uint64_t dv = smem_desc(smem_base, kChunkBytes, 1024, kSwizzle128B);
    const uint64_t dp = smem_desc(smem_base + kOffP, 16, 512, kSwizzle64B);
    // p_ok(j) stands for everything PV(j) needs: P(j) arrived and O rescaled
    // (warps 0-3, which saw p_full(j)), V(j)'s receive half landed and its
    // own half fenced into the async proxy (warp 9).
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int vs = j % kRecv, os = j % kOwn, slot = j % kPSlots;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.p_ok[slot], (j / kPSlots) & 1));
      TR_LAP(8, 0);  // PV issuer: waiting for p_ok
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t sv[2] = {static_cast<uint64_t>((kOffRecv + vs * kHalfBytes) >> 4),
                                static_cast<uint64_t>((kOffOwn + os * kHalfBytes) >> 4)};
        const uint64_t po = static_cast<uint64_t>((slot * kPSlotBytes) >> 4);
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
          for (int n = 0; n < 2; ++n)
            mma_ss(tbase + kColO + 256 * n, dp + po + ((32 * k) >> 4), dv + sv[n] + ((2048 * k) >> 4), id_o,
                   (j > 0 || k > 0) ? 1u : 0u);
        mma_commit_mc(&bar.v_free[vs], 0x3);
        mma_commit(&bar.own_free[os]);
        mma_commit_mc(&bar.p_free[slot], 0x3);
        mma_commit(&bar.pv_done[slot]);
        if (j == ntiles - 1) mma_commit(&bar.o_final);
      }
      __syncwarp();
      TR_LAP(8, 1);  // PV issuer: issuing
    }
    if (!ok) set_abort(bar, a.dev_error);
    if (lane == 0) mma_commit(&bar.fin[0]);
    __syncwarp();
    mbar_wait(&bar.fin[0], 0);
  } else if (!score && warp < 8) {
    const int q4 = warp & 3;
    const int h = q4 * 32 + lane;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(q4 * 32) << 16);
    bool ok = true;
    if (warp < 4) {
      // ----------------------------------------------- max tracking, rescale
      float m_prev = -INFINITY;
      for (int j = 0; j < ntiles; ++j) {
        const int slot = j % kPSlots;
        ok = __all_sync(0xffffffffu, mbar_wait_cluster(&bar.p_full[slot], (j / kPSlots) & 1));
        TR_LAP(9, 0);  // value warps 0-3: waiting for P
        if (!ok) break;
        // the slot's next fill (tile j + kPSlots) cannot start before PV(j)
        // frees it, and PV(j) waits for this warp's p_ok below
        if (warp == 0 && lane == 0) mbar_arrive_expect_tx(&bar.p_full[slot], kPTx);
        ++pdone;
        const float m_new = *reinterpret_cast<const volatile float*>(smem + kOffP + slot * kPSlotBytes + kPBytes + 4 * h);
        // a tile computed with m = -inf has P = 0 and leaves O as it is
        const bool need = m_new != m_prev && m_prev != -INFINITY && m_new != -INFINITY;
        if (__any_sync(0xffffffffu, need)) {
          // O holds PV(0..j-1): wait for PV(j-1), then scale this warp's rows.
          // PV(j - 1 - kPSlots) is complete (P(j) needed its slot), and PV(j)
          // cannot start before this warp's p_ok, so the parity is unambiguous.
          const int jp = j - 1;
          ok = __all_sync(0xffffffffu, mbar_wait(&bar.pv_done[jp % kPSlots], (jp / kPSlots) & 1));
          if (!ok) break;
          tc_fence_after();
          const float alpha = need ? ex2_approx(m_prev - m_new) : 1.f;
          for (int c = 0; c < 16; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_addr + kColO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_addr + kColO + 32 * c, o);
          }
          tmem_wait_st();
        }
        if (m_new != -INFINITY) m_prev = m_new;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.p_ok[slot]);
        TR_LAP(9, 1);  // value warps 0-3: max check / rescale
      }
    }
    // ------------------------------------------------------------ epilogue
    // warps 0-3 write value dims [0, 256), warps 4-7 dims [256, 512).  Each
    // 32-column block of a warp's 32 rows goes through a padded shared-memory
    // transpose (stage 0 is idle by now), so that every store instruction
    // writes 128 contiguous bytes of one O row.
    TR_MARK(9);
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar.o_final, 0) && mbar_wait_cluster(&bar.fin_l, 0));
    TR_LAP(9, 2);  // epilogue warps: waiting for the last PV
    if (ok) ok = !__any_sync(0xffffffffu, aborted(bar));
    if (!ok) {
      set_abort(bar, a.dev_error);
    } else {
      tc_fence_after();
      const float inv = *reinterpret_cast<const volatile float*>(smem + kOffFin + 4 * h);
      const int c0 = (warp >> 2) * 8;
      // 32 rows x 32 fp32 per block, rows 144 B apart (16-byte aligned; a
      // warp's 16-byte writes and reads then hit 4 banks groups at most)
      float* scr = reinterpret_cast<float*>(smem + kOffStages) + warp * (32 * 36);
      const int nrows = min(32, a.H - q4 * 32);
      for (int c = c0; c < c0 + 8; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + kColO + 32 * c, o);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<float4*>(scr + lane * 36 + 4 * k) =
              make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                          __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
        __syncwarp();
        if (!a.o_bf16) {
          // lane l: row 4 m + l / 8, columns 4 (l % 8) .. + 3 of the block
          float* orow0 = static_cast<float*>(a.O_dst) + (pair0 + q4 * 32) * kLatent;
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const int rr = 4 * m + (lane >> 3);
            if (rr < nrows)
              *reinterpret_cast<float4*>(orow0 + rr * kLatent + 32 * c + 4 * (lane & 7)) =
                  *reinterpret_cast<const float4*>(scr + rr * 36 + 4 * (lane & 7));
          }
        } else {
          // bf16 (round to nearest even), lane l: row 8 m + l / 4, columns
          // 8 (l % 4) .. + 7 of the block: 64 contiguous bytes per row
          __nv_bfloat16* orow0 = static_cast<__nv_bfloat16*>(a.O_dst) + (pair0 + q4 * 32) * kLatent;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int rr = 8 * m + (lane >> 2);
            if (rr < nrows) {
              const float4 x0 = *reinterpret_cast<const float4*>(scr + rr * 36 + 8 * (lane & 3));
              const float4 x1 = *reinterpret_cast<const float4*>(scr + rr * 36 + 8 * (lane & 3) + 4);
              __nv_bfloat162 b0 = __floats2bfloat162_rn(x0.x, x0.y), b1 = __floats2bfloat162_rn(x0.z, x0.w);
              __nv_bfloat162 b2 = __floats2bfloat162_rn(x1.x, x1.y), b3 = __floats2bfloat162_rn(x1.z, x1.w);
              *reinterpret_cast<uint4*>(orow0 + rr * kLatent + 32 * c + 8 * (lane & 3)) =
                  make_uint4(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1),
                             *reinterpret_cast<uint32_t*>(&b2), *reinterpret_cast<uint32_t*>(&b3));
            }
          }
        }
        __syncwarp();
      }
    }
  }

  // ------------------------------------------------------------- teardown
  TR_LAP(9, 3);  // epilogue (value warps 0-7), end of role for the others
  TR_DUMP();
  // the grid that consumes O_part / lse_part may start launching now; it
  // waits for this grid's completion before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const bool failed = aborted(bar);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer has issued everything it will send here
  if (failed && !score && threadIdx.x == 0) {
    // a failed unit may have left some of the score CTA's copies in flight
    // into the P slots: give each slot's next phase a short bounded wait
    for (int b = 0; b < kPSlots; ++b) {
      const int received = pdone > b ? (pdone - 1 - b) / kPSlots + 1 : 0;
      mbar_wait_cluster(&bar.p_full[b], received & 1, 1u << 16);
    }
  }
  if (warp == 10) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  TR_EXIT(unit);
}

// Launch order of the units (see launch_unit_order): one CTA; keys count
// into 33 buckets, then a stable scatter in chunks of 1024 units (rank in the
// warp by __match_any_sync, warps before this one by their bucket counts).
__global__ void __launch_bounds__(1024) unit_order_kernel(DecodeArgs a, int32_t units, int32_t* order) {
  __shared__ int32_t cnt[33], off[33];
  __shared__ int32_t wcnt[32][33];
  const int t = threadIdx.x, w = t >> 5, lane = t & 31;
  auto key_of = [&](int32_t u) -> int {
    const UnitCoords uc = unit_coords(a, u);
    const int r = uc.r, d = a.d0 + uc.dd, s = uc.s;
    const RowInfo ri = resolve_row(a.seq_lens, a.qsl, a.B, r, a.max_seq_len, a.max_q_len);
    const int32_t n = ri.padding ? 0 : local_len(ri.L, d, a.D, a.I);
    const int32_t lo = s * a.plan.chunk, hi = min(n, lo + a.plan.chunk);
    const int32_t tiles = lo < hi ? (hi - lo + kTile - 1) / kTile : 0;
    return tiles == 0 ? 0 : 32 - __clz(tiles);  // 1 + floor(log2 tiles)
  };
  if (t < 33) cnt[t] = 0;
  __syncthreads();
  for (int32_t u = t; u < units; u += 1024) atomicAdd(&cnt[key_of(u)], 1);
  __syncthreads();
  if (t == 0) {
    int32_t acc = 0;
    for (int k = 32; k >= 0; --k) { off[k] = acc; acc += cnt[k]; }
  }
  __syncthreads();
  for (int32_t base = 0; base < units; base += 1024) {
    for (int i = t; i < 32 * 33; i += 1024) (&wcnt[0][0])[i] = 0;
    __syncthreads();
    const int32_t u = base + t;
    const int k = u < units ? key_of(u) : -1;
    const unsigned same = __match_any_sync(0xffffffffu, k);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (k >= 0 && rank == 0) wcnt[w][k] = __popc(same);
    __syncthreads();
    if (k >= 0) {
      int32_t pos = off[k] + rank;
      for (int v = 0; v < w; ++v) pos += wcnt[v][k];
      order[pos] = u;
    }
    __syncthreads();
    if (t < 33) {
      int32_t add = 0;
      for (int v = 0; v < 32; ++v) add += wcnt[v][t];
      off[t] += add;
    }
    __syncthreads();
  }
}

cudaLaunchConfig_t launch_config(int64_t units, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * units));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

namespace {
// Per-device one-time set-up of the tensor-core decode: its shared-memory
// opt-in and the number of its clusters that fit on the device at once.  One
// entry per device, behind a mutex, so that concurrent host threads and
// alternating devices always size the split plan from the same count, and a
// launch (possibly inside a stream capture) makes no attribute call.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
int g_resident[kMaxDevices] = {};  // 0: not yet set up

int setup_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  if (dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_resident[dev] > 0) return g_resident[dev];
  if (cudaFuncSetAttribute(decode_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
          cudaSuccess ||
      cudaFuncSetAttribute(decode_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
          cudaSuccess) { cudaGetLastError(); return 0; }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(1, nullptr, attr);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, decode_tc_kernel<false>, &cfg) != cudaSuccess || clusters <= 0) {
    cudaGetLastError();
    return 0;
  }
  g_resident[dev] = 2 * clusters;
  return g_resident[dev];
}
}  // namespace

int decode_tc_resident_ctas() {
  // CTAs of the tensor-core decode that fit on the current device at once
  // (1 per SM by shared memory; clusters of two must sit in one GPC).
  return setup_current_device();
}

cudaError_t launch_unit_order(const DecodeArgs& a, int32_t units, int32_t* order, cudaStream_t st) {
  if (units <= 0) return cudaSuccess;
  unit_order_kernel<<<1, 1024, 0, st>>>(a, units, order);
  return cudaGetLastError();
}

// (Cache rows are addressed in 31 bits: a cache of 2^31 rows would be 2.5 TB.)
bool decode_tc_supported(const DecodeArgs& a) {
  return a.H <= 128 && (a.plan.chunk % kTile) == 0 &&
         static_cast<int64_t>(a.num_blocks) * a.block_size <= 0x7fffffffLL;
}

#ifdef DCP_DEBUG_WAITS
// Debug builds only: the waits that gave up ([count] then [256][4]: barrier
// shared address, parity, CTA, thread).
extern "C" int dcp_wait_log_fetch(void* dst, size_t bytes) {
  unsigned int n = 0;
  if (cudaMemcpyFromSymbol(&n, sm100::g_dcp_wait_count, sizeof(n)) != cudaSuccess) return -1;
  if (bytes < 4) return -1;
  memcpy(dst, &n, 4);
  size_t rest = bytes - 4;
  if (rest > sizeof(sm100::g_dcp_wait_log)) rest = sizeof(sm100::g_dcp_wait_log);
  return static_cast<int>(cudaMemcpyFromSymbol(static_cast<char*>(dst) + 4, sm100::g_dcp_wait_log, rest));
}
#endif

#ifdef DCP_TRACE
// Traced builds only: copy the counters and the per-CTA timeline of the last
// launch to the host.
extern "C" int dcp_trace_fetch(void* dst, size_t bytes) {
  if (bytes > sizeof(g_dcp_trace)) bytes = sizeof(g_dcp_trace);
  return static_cast<int>(cudaMemcpyFromSymbol(dst, g_dcp_trace, bytes));
}
extern "C" int dcp_timeline_fetch(void* dst, size_t bytes) {
  if (bytes > sizeof(g_dcp_timeline)) bytes = sizeof(g_dcp_timeline);
  return static_cast<int>(cudaMemcpyFromSymbol(dst, g_dcp_timeline, bytes));
}
#endif

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
  if (!decode_tc_supported(a)) return cudaErrorInvalidValue;
  if (setup_current_device() <= 0) return cudaErrorInvalidDevice;
  const int64_t units = static_cast<int64_t>(a.T) * a.Dn * a.plan.splits;
  if (2 * units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(units, st, attr);
  return a.kv_fp8 ? cudaLaunchKernelEx(&cfg, decode_tc_kernel<true>, a) : cudaLaunchKernelEx(&cfg, decode_tc_kernel<false>, a);
}

}  // namespace dcp
