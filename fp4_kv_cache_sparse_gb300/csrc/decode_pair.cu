// decode_pair.cu -- token-sparse MLA decode for 128 query heads on a cluster of
// two CTAs that split the 512 latent dims (sm_103a: tcgen05 + TMEM + TMA +
// distributed shared memory).
//
// What it computes is the same as decode.cu ("flops/flashmla-decode-fp8-fp4-kv",
// "Arithmetic intensity" and "Workarounds"; "deepseek-ai/FlashMLA", "How to use
// it"), for an FP8 main cache without an extra cache.  The layout differs:
// heads are the MMA's M dimension (all 128 of them).  O for 128 heads x 512
// dims would fill all of TMEM, so CTA c of the pair owns dims [256c, 256c+256):
// its half of every record, of Q (kept in TMEM as the A operand of
// S = Q K^T), of the bf16 tile and of O.  Each CTA's S is a partial sum over
// its dims.  A scheduled 128-token tile is processed as two 64-token
// sub-tiles, so that S fits TMEM twice next to O and Q: the tensor core
// computes the next sub-tile's S while the softmax warps work on the current
// one.  CTA c computes the softmax of token quarter c of every sub-tile
// (tokens 32c .. 32c+31) for all heads: it sends the peer its partial scores
// of the peer's quarter and receives the peer's for its own (bulk
// asynchronous copies between the two shared memories, completing on the
// receiver's mbarrier), the two CTAs swap per-head tile maxima so that they
// keep identical running maxima (and rescale factors), and each sends the
// other its part of P, so both hold all of P for their O += P V.  P and the
// received partial scores are double-buffered by sub-tile parity, so a
// sub-tile's softmax does not wait for the previous sub-tile's PV; the bf16
// tile has four buffers, as a buffer is held from its dequantization to the
// end of the PV that reads it.  One thread issues each product as soon as
// its inputs are ready (O += P V as one 128x256x16 product per 16 tokens).  Records reach shared memory by TMA row gathers
// (tile::gather4, 4 tokens per instruction, 256 bytes of a record per row)
// into a 3-slot staging ring, so the dequantizing warps never have global
// loads in flight when they publish a slot.  Outputs (and split partials)
// leave by TMA tensor stores of 32-row x 32-dim blocks staged in the idle P
// buffers.
//
// Warps: 0-7 softmax (two per TMEM lane quadrant, one per 16-token column
// half of the quarter), 8-11 dequant, 12 loader (indices, validity mask,
// scales, TMA row gathers), 13 tensor-core issuer.
#include <cstdint>
#include <cuda.h>

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kPThreads = 448;
constexpr int kHeads = 128;
constexpr int kHalf = 256;
constexpr int kStgSlots = 3;
constexpr int kKvBufs = 4;
constexpr int kProdWarps = 4;
constexpr int kSoftThreads = 256;
constexpr int kLoaderWarp = 12;
constexpr int kIssueWarp = 13;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLazy = 8.0f;
constexpr uint32_t kXWarpBytes = 32 * 64;       // one softmax warp's 32 heads x 16 tokens of fp32 scores
constexpr uint32_t kPWarpBytes = 32 * 32;       // one softmax warp's 32 heads x 16 tokens of bf16 P
constexpr uint32_t kPInBytes = 8 * kPWarpBytes;  // the peer's quarter of P

struct PairSmem {
  static constexpr int kKV = 0;                  // 4 buffers x 4 chunks x [64 tokens x 128 B], SW128
  static constexpr int kP = kKV + kKvBufs * 32768;  // 2 buffers (sub-tile parity) x 4 chunks (16 tokens each:
                                                 // K steps of O += P V) x [128 heads x 32 B] bf16, SW32, so
                                                 // each softmax warp's P rows are one contiguous 1 KB block
  static constexpr int kX = kP + 2 * 16384;      // 2 buffers x 8 warps x [32 heads x 16 tokens] fp32 from the
                                                 // peer, SW64 units; a sub-tile's outgoing partial scores are
                                                 // staged in the other parity's buffer
  static constexpr int kStg = kX + 2 * 16384;    // 3 slots x [32 tokens x 256 B] raw e4m3 (this CTA's dims)
  static constexpr int kScl = kStg + kStgSlots * 8192;  // 2 x [4][32] x 8 B e8m0 scales of this CTA's dims
                                                        // (token 4l + j of a 128-token tile at [j][l])
  static constexpr int kBar = kScl + 2 * 1024;   // 64 mbarriers
  static constexpr int kMask = kBar + 64 * 8;    // [2][4] u32 validity bits
  static constexpr int kMaxIn = kMask + 32;      // [4 quadrants][2 column halves][32] f32 tile maxima from the peer
  static constexpr int kMaxOut = kMaxIn + 1024;  // the same, this CTA's, for the peer
  static constexpr int kStats = kMaxOut + 1024;  // [2 parities][2 column halves][128] f32 row sums from the peer
  static constexpr int kStatsOut = kStats + 2048;  // [2 column halves][128] f32 row sums for the peer
  static constexpr int kScalar = kStatsOut + 1024;  // tmem slot, abort flag
  static constexpr int kEnd = kScalar + 16;
  static constexpr int kAlloc = kEnd + 1024;
};
static_assert(PairSmem::kAlloc <= 227 * 1024, "dynamic shared memory of one CTA");

// mbarrier indices; each range is as long as the count that indexes it.
enum PairBar : int {
  bStgFull = 0, bStgFree = bStgFull + kStgSlots, bSclFull = bStgFree + kStgSlots, bSclFree = bSclFull + 2,
  bMaskFull = bSclFree + 2, bMaskFree = bMaskFull + 2, bKvFull = bMaskFree + 2, bKvFree = bKvFull + kKvBufs,
  bQFull = bKvFree + kKvBufs, bSFull = bQFull + 1 /* [2 S buffers] */, bSUsed = bSFull + 2,
  bPMine2 = bSUsed + 2 /* [2] by sub-tile parity */, bPIn = bPMine2 + 2 /* [2 P buffers] */, bPvDone = bPIn + 2,
  bOReady = bPvDone + 2, bStatsIn = bOReady + 1 /* [2] */, bDrain = bStatsIn + 2,
  bXFull = bDrain + 1 /* [2 X buffers][8 warps] */, bMaxFull = bXFull + 16 /* [4 quadrants] */,
  kNumPairBars = bMaxFull + 4
};
static_assert(kNumPairBars <= 64, "the mbarrier area holds 64 barriers");

// TMEM columns: S [0, 128) as two 64-column buffers, O [128, 384), Q [384, 512)
// (this CTA's 256 dims of the query token as packed bf16 pairs: the A operand
// of S = Q K^T).
constexpr uint32_t kColS = 0, kColO = 128, kColQ = 384;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_of(uint32_t local, uint32_t peer) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(peer));
  return r;
}
// Bulk copy of this CTA's shared memory into the peer's, completing on the
// peer's mbarrier (transaction bytes).
__device__ __forceinline__ void bulk_to_peer(uint32_t dst_peer, const void* src, uint32_t bytes, uint32_t bar_peer) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_peer),
               "r"(smem_u32(src)), "r"(bytes), "r"(bar_peer)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most one of this thread's bulk groups still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Waits until every bulk group of this thread has completed (writes included).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Tiled TMA store of a shared-memory box to global coordinates (x, y).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_commit_and_wait_read() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// 32 bytes from global memory (read-only path); p must be 32-byte aligned.
__device__ __forceinline__ void ldg_v8(const void* p, uint32_t* r) {
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}

// Non-blocking test of a phase's completion.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
// Four rows (tokens) of a 2-D byte tensor, x bytes in, into consecutive rows of dst.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, int x, int r0, int r1, int r2, int r3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16: A is M rows (lanes) x K
// columns of packed bf16 pairs.  One elected lane of a converged warp issues.
__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ss_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
// Bounded wait used when the CTA is about to end: it ignores the abort flag
// (products already issued must complete before TMEM goes away) but gives
// up after its own limit.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, int32_t* d_error) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63) == 63 && global_timer_ns() - t0 > kWaitNs) {
      if (d_error) atomicOr(d_error, MLA_DEVERR_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%"
      "29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%"
      "30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

struct PSpan {
  int64_t g_begin, g_end;
  int first_local_split;
  bool ok;
};

__device__ __forceinline__ PSpan pair_span(const DecodeParams& p, int part) {
  PSpan s;
  const int32_t* e = p.sched + static_cast<int64_t>(part) * MLA_SCHED_INTS;
  s.g_begin = e[0];
  s.g_end = e[1];
  s.first_local_split = e[2];
  const int64_t G = static_cast<int64_t>(p.nq) * p.T;
  s.ok = s.g_begin >= 0 && s.g_begin <= s.g_end && s.g_end <= G && s.first_local_split >= 0;
  if (!s.ok) s.g_begin = s.g_end = 0;
  return s;
}

// kRope: query tokens of one split leave as FP8 records after the
// conjugate rotary embedding (the fused epilogue) instead of bf16 rows; a
// separate instantiation, so that the bf16 kernel carries none of it.
template <bool kRope>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
    sparse_decode_pair_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kv_map,
                              const __grid_constant__ CUtensorMap out_map, const __grid_constant__ CUtensorMap ws_map) {
  using L = PairSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKV = smem + L::kKV;
  uint8_t* sP = smem + L::kP;
  uint8_t* sX = smem + L::kX;
  uint8_t* sStg = smem + L::kStg;
  uint8_t* sScl = smem + L::kScl;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* sMask = reinterpret_cast<uint32_t*>(smem + L::kMask);
  float* sMaxIn = reinterpret_cast<float*>(smem + L::kMaxIn);
  float* sMaxOut = reinterpret_cast<float*>(smem + L::kMaxOut);
  float* sStats = reinterpret_cast<float*>(smem + L::kStats);
  float* sStatsOut = reinterpret_cast<float*>(smem + L::kStatsOut);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kScalar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kScalar + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t c = cluster_rank();
  const uint32_t peer = c ^ 1u;
  const int part = blockIdx.x >> 1;

  if (tid == 0) {
    for (int i = 0; i < kStgSlots; ++i) {
      mbar_init(&bars[bStgFull + i], 1);
      mbar_init(&bars[bStgFree + i], kProdWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[bSclFull + i], 1);
      mbar_init(&bars[bSclFree + i], kProdWarps);
      mbar_init(&bars[bMaskFull + i], 1);
      mbar_init(&bars[bMaskFree + i], kSoftThreads / 32);  // per-warp arrivals (lane 0 after __syncwarp)
      mbar_init(&bars[bStatsIn + i], 1);
      mbar_init(&bars[bSFull + i], 1);
      mbar_init(&bars[bSUsed + i], kSoftThreads / 32);
    }
    for (int b = 0; b < kKvBufs; ++b) {
      mbar_init(&bars[bKvFull + b], 2 * kProdWarps);  // two 32-token slots per 64-token sub-tile
      mbar_init(&bars[bKvFree + b], 1);
    }
    mbar_init(&bars[bQFull], kSoftThreads / 32);  // one arrival per softmax warp, after its lanes' writes
    for (int b = 0; b < 2; ++b) mbar_init(&bars[bPMine2 + b], kSoftThreads / 32);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[bPIn + b], 1);
      mbar_init(&bars[bPvDone + b], 1);
    }
    mbar_init(&bars[bOReady], 1);
    mbar_init(&bars[bDrain], 1);
    for (int w = 0; w < 16; ++w) mbar_init(&bars[bXFull + w], 1);
    for (int w = 0; w < 4; ++w) mbar_init(&bars[bMaxFull + w], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers exist before anyone arrives on them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const PSpan span = pair_span(p, part);
  if (!span.ok && tid == 0 && c == 0 && p.d_error) atomicOr(p.d_error, MLA_DEVERR_BAD_METADATA);

  if (warp == kLoaderWarp) {
    // ------------------------------------------------------------------
    // Loader: indices -> validity mask; this CTA's 8 scale bytes of every
    // record by plain loads, one tile ahead; TMA row gathers of the record
    // halves (256 bytes per token), 32 tokens per staging slot.
    // Lane l covers tokens 4l .. 4l+3 of a tile.
    // ------------------------------------------------------------------
    uint32_t n_tile = 0, n_chunk = 0;
    auto raw_ids = [&](int64_t g, int32_t (&id)[4]) {
      const int qidx = static_cast<int>(g / p.T);
      const int t = static_cast<int>(g - static_cast<int64_t>(qidx) * p.T);
      const int32_t* ids = p.idx + static_cast<int64_t>(qidx) * p.topk;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int slot = t * kTile + 4 * lane + j;
        id[j] = slot < p.topk ? __ldg(ids + slot) : -1;
      }
    };
    auto valid_id = [&](int32_t id) { return id >= 0 && static_cast<int64_t>(id) < p.pool_tokens; };
    auto load_scales = [&](const int32_t (&id)[4], uint2 (&sc)[4]) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        sc[j] = valid_id(id[j]) ? __ldg(reinterpret_cast<const uint2*>(p.kv + static_cast<int64_t>(id[j]) * kRecFp8 +
                                                                      kD + 8 * c))
                                : make_uint2(0u, 0u);
    };
    int32_t cur[4] = {-1, -1, -1, -1}, nxt[4] = {-1, -1, -1, -1};
    uint2 sc_cur[4] = {}, sc_nxt[4] = {};
    if (span.g_begin < span.g_end) raw_ids(span.g_begin, cur);
    if (span.g_begin + 1 < span.g_end) raw_ids(span.g_begin + 1, nxt);
    load_scales(cur, sc_cur);
    for (int64_t g = span.g_begin; g < span.g_end; ++g, ++n_tile) {
      // Validity; rows for the gathers (-1 = outside the tensor: zero fill).
      int32_t row[4];
      uint32_t vbits[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int32_t id = cur[j];
        const bool valid = valid_id(id);
        if (!valid && id != -1 && c == 0 && p.d_error) atomicOr(p.d_error, MLA_DEVERR_BAD_INDEX);
        row[j] = valid ? id : -1;
        vbits[j] = __ballot_sync(0xFFFFFFFFu, valid);
      }
      // The next tile's scales and the indices of the tile after it go out
      // now, a whole tile of gathers ahead of their use.
      load_scales(nxt, sc_nxt);
      int32_t nxt2[4] = {-1, -1, -1, -1};
      if (g + 2 < span.g_end) raw_ids(g + 2, nxt2);
      const uint32_t mp = n_tile & 1;
      if (n_tile >= 2) mbar_wait(&bars[bSclFree + mp], ((n_tile >> 1) - 1) & 1, abort_flag, p.d_error, kWaitNs);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint2*>(sScl + mp * 1024 + (32 * j + lane) * 8) = sc_cur[j];
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[bSclFull + mp]);
        if (n_tile >= 2) mbar_wait(&bars[bMaskFree + mp], ((n_tile >> 1) - 1) & 1, abort_flag, p.d_error, kWaitNs);
#pragma unroll
        for (int j = 0; j < 4; ++j) sMask[mp * 4 + j] = vbits[j];
        mbar_arrive(&bars[bMaskFull + mp]);
      }
#pragma unroll 1
      for (int k = 0; k < 4; ++k, ++n_chunk) {
        const uint32_t slot = n_chunk % kStgSlots, use = n_chunk / kStgSlots;
        if (lane == 0) {
          if (use > 0) mbar_wait(&bars[bStgFree + slot], (use - 1) & 1, abort_flag, p.d_error, kWaitNs);
          mbar_expect_tx(&bars[bStgFull + slot], 32 * 256);
        }
        __syncwarp();
        if ((lane >> 3) == k)
          tma_gather4(sStg + slot * 8192 + (lane & 7) * 1024, &kv_map, static_cast<int>(c) * kHalf, row[0], row[1],
                      row[2], row[3], &bars[bStgFull + slot]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        cur[j] = nxt[j];
        nxt[j] = nxt2[j];
        sc_cur[j] = sc_nxt[j];
      }
    }
    // The gathers of the last slots land before this CTA's shared memory
    // goes away, even after a timeout (normally they completed long ago).
    if (lane == 0) {
      for (uint32_t k = 0; k < kStgSlots && k < n_chunk; ++k) {
        const uint32_t i = n_chunk - 1 - k;
        mbar_wait_drain(&bars[bStgFull + i % kStgSlots], (i / kStgSlots) & 1, p.d_error);
      }
    }
    __syncwarp();
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------------
    // Dequantizers: staging slot (32 tokens x this CTA's 256 dims, raw e4m3)
    // + scales -> bf16 rows of a sub-tile buffer (two slots per 64-token
    // sub-tile, four buffers in turn).  Lane L (0..127) handles items
    // L + 128r (r = 0..3) of a slot; item i is token i >> 4, 16-dim segment
    // i & 15.
    // ------------------------------------------------------------------
    const int L = tid - 256;
    uint32_t n_tile = 0, n_chunk = 0, n_sub = 0;
    for (int64_t g = span.g_begin; g < span.g_end; ++g, ++n_tile) {
      const uint32_t mp = n_tile & 1;
      mbar_wait(&bars[bSclFull + mp], (n_tile >> 1) & 1, abort_flag, p.d_error, kWaitNs);
      const uint8_t* scl = sScl + mp * 1024;
#pragma unroll 1
      for (int sub = 0; sub < 2; ++sub, ++n_sub) {
        const uint32_t buf = n_sub % kKvBufs, use = n_sub / kKvBufs;
        if (use > 0) mbar_wait(&bars[bKvFree + buf], (use - 1) & 1, abort_flag, p.d_error, kWaitNs);
        uint8_t* tile = sKV + buf * 32768;
#pragma unroll 1
        for (int kk = 0; kk < 2; ++kk, ++n_chunk) {
          const int k = 2 * sub + kk;  // slot of the 128-token tile
          const uint32_t slot = n_chunk % kStgSlots, suse = n_chunk / kStgSlots;
          mbar_wait(&bars[bStgFull + slot], suse & 1, abort_flag, p.d_error, kWaitNs);
          const uint8_t* stg = sStg + slot * 8192;
#pragma unroll 1
          for (int rb = 0; rb < 4; rb += 4) {
            uint4 raw[4];
            uint32_t sb[4];
            bool big = false;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int item = L + 128 * (rb + r);
              const int tt = item >> 4, s = item & 15;
              raw[r] = *reinterpret_cast<const uint4*>(stg + item * 16);
              const int T = 32 * k + tt;  // scales of token T = 4l + j sit at [j][l]
              sb[r] = scl[(32 * (T & 3) + (T >> 2)) * 8 + (s >> 1)];
              big |= sb[r] > 142u;
            }
            const bool any_big = __any_sync(0xFFFFFFFFu, big);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int item = L + 128 * (rb + r);
              const int t = 32 * kk + (item >> 4), s = item & 15;  // row of the sub-tile
              uint32_t o[8];
              if (!any_big)
                dequant_fp8_16_small_scale(raw[r], sb[r], o);
              else
                dequant_fp8_16(raw[r], sb[r], o);
              uint8_t* chunk = tile + (s >> 2) * 8192;
              // Segments of odd 64-dim chunks store their upper 16-byte unit
              // first, so that the 8 lanes of each quarter-warp store to 8
              // distinct bank groups.
              const bool odd = (s >> 2) & 1;
              const int u = 2 * (s & 3);
              const uint4 lo = make_uint4(o[0], o[1], o[2], o[3]), hi = make_uint4(o[4], o[5], o[6], o[7]);
              *reinterpret_cast<uint4*>(chunk + swz<128>(t * 128 + (u + odd) * 16)) = odd ? hi : lo;
              *reinterpret_cast<uint4*>(chunk + swz<128>(t * 128 + (u + !odd) * 16)) = odd ? lo : hi;
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bars[bKvFull + buf]);
            mbar_arrive(&bars[bStgFree + slot]);
            if (k == 3) mbar_arrive(&bars[bSclFree + mp]);
          }
        }
      }
    }
  } else if (warp == kIssueWarp) {
    // ------------------------------------------------------------------
    // Tensor-core issue.  The whole warp runs the loop (lane 0 tests the
    // barriers and broadcasts what it saw, so the warp stays converged) and
    // one elected lane issues each product: per 64-token sub-tile, S = Q K^T
    // (A = Q in TMEM, into the S buffer of the sub-tile's parity), O += P V
    // over this CTA's token quarter once its P is written and over the
    // peer's once the peer's P has landed, each as soon as it can go.
    // ------------------------------------------------------------------
    constexpr uint32_t idesc_qk = make_idesc_bf16(128, 64, false, false);
    constexpr uint32_t idesc_pv = make_idesc_bf16(128, 256, false, true);
    const uint32_t kv_base = smem_u32(sKV), p_base = smem_u32(sP);
    const uint32_t tS = tmem + kColS, tO = tmem + kColO, tQ = tmem + kColQ;
    uint32_t n_sub = 0, n_seg = 0;
    bool issued = false;
    auto test = [&](int bar, uint32_t parity) {
      int ok = 0;
      if (lane == 0) ok = mbar_test(&bars[bar], parity);
      return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
    };
    auto issue_qk = [&](uint32_t nt) {
      const uint32_t buf = nt % kKvBufs, sb = nt & 1;
      // B descriptor of the first K step; later steps only move the start
      // address (the 14-bit field cannot carry: shared memory ends below
      // 256 KB).
      const uint64_t b0 = make_smem_desc(kv_base + buf * 32768, 16, 1024, kSwizzle128);
      const uint32_t d = tS + 64 * sb;
      // A loop over the four 64-dim chunks, not unrolled: the issue paced
      // this way measured faster (~1 % on the 128-head shapes) than all
      // 16 products back to back or a loop of 2 or 1.
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_elect(d, tQ + k * 32 + kk * 8, b0 + ((k * 8192 + kk * 32) >> 4), idesc_qk, (k | kk) != 0);
      }
      commit_elect(&bars[bSFull + sb]);
    };
    // O += P V over the 16-token K steps q0, q0+1 (this CTA's quarter or
    // the peer's) of sub-tile buffer buf: one N = 256 product per step, all
    // four 64-dim chunks of this CTA's V at once, so P is read once.
    auto issue_pv = [&](uint32_t buf, uint32_t pb, int q0, bool init) {
      const uint64_t a0 = make_smem_desc(p_base + pb * 16384 + q0 * 4096, 16, 256, kSwizzle32);
      const uint64_t b0 = make_smem_desc(kv_base + buf * 32768 + q0 * 2048, 8192, 1024, kSwizzle128);
      mma_ss_elect(tO, a0, b0, idesc_pv, !init);
      mma_ss_elect(tO, a0 + (4096 >> 4), b0 + (2048 >> 4), idesc_pv, 1);
    };
    for (int64_t g = span.g_begin; g < span.g_end;) {
      const int qidx = static_cast<int>(g / p.T);
      const int64_t seg_end = min(span.g_end, static_cast<int64_t>(qidx + 1) * p.T);
      const uint32_t seg_subs = static_cast<uint32_t>(2 * (seg_end - g));
      const uint32_t base = n_sub;
      // Q of this query token is in TMEM once the softmax warps have
      // written it (after the previous token's epilogue).
      mbar_wait(&bars[bQFull], n_seg & 1, abort_flag, p.d_error, kWaitNs);
      __syncwarp();
      tc_fence_after();
      issued = true;
      // Issue each product of the segment as soon as its inputs are ready:
      // the second half of O += P V first (it frees a tile buffer for the
      // dequantizers), then the first half, then the next S = Q K^T (its S
      // buffer released by the softmax two sub-tiles back, its tile in
      // shared memory), so that the tensor core works during the softmax.
      uint32_t qk = 0, pva = 0, pvb = 0;
      uint64_t idle_since = 0;
      uint32_t idle_it = 0;
      bool stop = false;
      while (pvb < seg_subs && !stop) {
        bool progress = false;
        if (pvb < pva) {
          const uint32_t n = base + pvb, pb = n & 1;
          if (test(bPIn + pb, (n >> 1) & 1)) {
            tc_fence_after();
            issue_pv(n % kKvBufs, pb, 2 * static_cast<int>(peer), false);
            commit_elect(&bars[bKvFree + n % kKvBufs]);
            commit_elect(&bars[bPvDone + pb]);
            if (pvb + 1 == seg_subs) commit_elect(&bars[bOReady]);
            ++pvb;
            progress = true;
          }
        }
        if (pva < qk) {
          const uint32_t n = base + pva;
          if (test(bPMine2 + (n & 1), (n >> 1) & 1)) {
            tc_fence_after();
            issue_pv(n % kKvBufs, n & 1, 2 * static_cast<int>(c), pva == 0);
            ++pva;
            progress = true;
          }
        }
        if (qk < seg_subs && qk < pva + 2) {
          const uint32_t n = base + qk, buf = n % kKvBufs;
          if ((n < 2 || test(bSUsed + (n & 1), ((n - 2) >> 1) & 1)) && test(bKvFull + buf, (n / kKvBufs) & 1)) {
            tc_fence_after();
            issue_qk(n);
            ++qk;
            progress = true;
          }
        }
        if (progress) {
          idle_it = 0;
        } else {
          __nanosleep(32);
          // The wait limit applies to each stretch without progress; the
          // clock is first read 64 idle polls into a stretch, so that the
          // short stretches between products cost no timer reads.
          if ((++idle_it & 63) == 0) {
            int quit = 0;
            if (lane == 0) {
              const uint64_t now = global_timer_ns();
              if (idle_it == 64) idle_since = now;
              if (*abort_flag) {
                quit = 1;
              } else if (now - idle_since > kWaitNs) {
                *abort_flag = 1;
                if (p.d_error) atomicOr(p.d_error, MLA_DEVERR_TIMEOUT);
                quit = 1;
              }
            }
            stop = __shfl_sync(0xFFFFFFFFu, quit, 0) != 0;
          }
        }
      }
      n_sub = base + seg_subs;
      g = seg_end;
      ++n_seg;
      if (stop) break;
    }
    if (issued) {
      // Every product issued completes before TMEM is released, even after
      // a timeout (this wait ignores the abort flag; it has its own bound).
      commit_elect(&bars[bDrain]);
      __syncwarp();
      mbar_wait_drain(&bars[bDrain], 0, p.d_error);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------
    // Softmax warps 0-7.  Warp w serves the 32 heads of TMEM lane quadrant
    // qd = w & 3 (lane <-> head 32 qd + lane <-> TMEM lane) and 16 of the 32
    // tokens of each quarter (ch = w >> 2), so two warps share each head.
    // This CTA owns the softmax of quarter c of every sub-tile: each warp
    // sends its 16 columns of the peer's quarter of the partial scores to the
    // peer's same warp and receives the peer's for its columns of this
    // quarter; per-head tile maxima of both warps of a quadrant are swapped
    // with the peer so both CTAs keep identical running maxima; each warp's
    // P (its 32 heads x 16 tokens) travels to the peer, so both hold all of
    // P for PV.
    // ------------------------------------------------------------------
    const int qd = warp & 3, ch = warp >> 2;
    const int i = 32 * qd + lane;  // head
    const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
    const uint32_t tS = tmem + lane_base + kColS, tO = tmem + lane_base + kColO, tQ = tmem + lane_base + kColQ;
    const int pair_bar = 2 + qd;  // named barrier of the two warps of quadrant qd
    uint32_t n_tile = 0, n_sub = 0, n_seg = 0;
    float m = -INFINITY, l = 0.f;  // running max (shared by both CTAs) and this warp's part of the row sum
    // Q row i of query token qx, dims [128 ch, 128 ch + 128) of my half, into
    // TMEM as packed bf16 pairs (columns 64 ch .. 64 ch + 63 of the Q area).
    auto q_src = [&](int qx) {
      return reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(qx) * kHeads + i) * kD +
                                            static_cast<int>(c) * kHalf + ch * 128);
    };
    // Each lane's rows start on 256-byte boundaries of q, so with q 32-byte
    // aligned the row goes in 32-byte loads (half the requests of 16-byte
    // ones); otherwise in 16-byte loads.
    const bool q_al32 = (reinterpret_cast<uintptr_t>(p.q) & 31) == 0;
    // FP8 records (528 bytes, a multiple of 16) in 16-byte pieces when the
    // destination allows, else in 4-byte words.
    const bool rope_al16 = (reinterpret_cast<uintptr_t>(p.rope_out) & 15) == 0;
    auto load_q = [&](int qx) {
      const uint4* src = q_src(qx);
#pragma unroll 1
      for (int j = 0; j < 2; ++j) {
        uint32_t v[32];
        if (q_al32) {
#pragma unroll
          for (int u = 0; u < 4; ++u) ldg_v8(src + j * 8 + 2 * u, v + 8 * u);
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 w = __ldg(src + j * 8 + u);
            v[4 * u] = w.x;
            v[4 * u + 1] = w.y;
            v[4 * u + 2] = w.z;
            v[4 * u + 3] = w.w;
          }
        }
        tmem_st32(tQ + 64 * ch + 32 * j, v);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[bQFull]);
    };
    if (span.g_begin < span.g_end) load_q(static_cast<int>(span.g_begin / p.T));
    for (int64_t g = span.g_begin; g < span.g_end;) {
      const int qidx = static_cast<int>(g / p.T);
      const int64_t seg_end = min(span.g_end, static_cast<int64_t>(qidx + 1) * p.T);
      const int64_t seg_begin = g;
      if (warp == 0 && lane == 0) mbar_expect_tx(&bars[bStatsIn + (n_seg & 1)], 1024);
      for (; g < seg_end; ++g, ++n_tile) {
        if (g + 1 == seg_end && seg_end < span.g_end) {
          // The next query token's Q rows into L2 now, two sub-tiles before
          // they are loaded.
          const uint4* nq = q_src(qidx + 1);
          asm volatile("prefetch.L2 [%0];" ::"l"(nq));
          asm volatile("prefetch.L2 [%0];" ::"l"(nq + 8));
        }
        // Validity of the 128-token tile: bit b of word e covers token 4b + e.
        const uint32_t mp = n_tile & 1;
        mbar_wait(&bars[bMaskFull + mp], (n_tile >> 1) & 1, abort_flag, p.d_error, kWaitNs);
        uint32_t mkw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) mkw[e] = sMask[mp * 4 + e];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[bMaskFree + mp]);
#pragma unroll 1
        for (int sub = 0; sub < 2; ++sub, ++n_sub) {
          const uint32_t sb = n_sub & 1, pb = n_sub & 1;  // S, P and X buffers of this sub-tile
          const uint32_t tSb = tS + 64 * sb;
          uint8_t* sPb = sP + pb * 16384;
          const uint8_t* sXw = sX + pb * 16384 + warp * 2048;
          // This warp's P rows: chunk 2c + ch (its 16 tokens) of the P buffer.
          uint8_t* sPw = sPb + (2 * static_cast<int>(c) + ch) * 4096;
          // Outgoing staging: this warp's block of the other parity's X
          // buffer.  The peer's partial scores of the next sub-tile land
          // there only after this sub-tile's copy has reached the peer.
          uint8_t* stg = sX + (pb ^ 1) * 16384 + warp * 2048;
          if (lane == 0) {
            mbar_expect_tx(&bars[bXFull + 8 * pb + warp], kXWarpBytes);
            if (ch == 0) mbar_expect_tx(&bars[bMaxFull + qd], 256);
          }
          mbar_wait(&bars[bSFull + sb], (n_sub >> 1) & 1, abort_flag, p.d_error, kWaitNs);
          // This warp's copies of earlier sub-tiles (out of this staging
          // block two sub-tiles back, of P and of maxima) are read.
          if (lane == 0) bulk_wait_read();
          __syncwarp();
          tc_fence_after();
          // 1. My 16 columns of the peer's quarter of the partial scores,
          //    pre-scaled, to my staging block and on to the peer's same warp.
          {
            uint32_t v[16];
            tmem_ld16(tSb + 32 * peer + 16 * ch, v);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4*>(stg + swz<64>(lane * 64 + u * 16)) =
                  make_uint4(__float_as_uint(__uint_as_float(v[4 * u]) * p.scale_log2),
                             __float_as_uint(__uint_as_float(v[4 * u + 1]) * p.scale_log2),
                             __float_as_uint(__uint_as_float(v[4 * u + 2]) * p.scale_log2),
                             __float_as_uint(__uint_as_float(v[4 * u + 3]) * p.scale_log2));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // The peer's X block of this warp and parity is free: the
            // peer's same warp read it (two sub-tiles back) before sending
            // its tile maxima of the previous sub-tile, which this warp has
            // received.
            bulk_to_peer(peer_of(smem_u32(sXw), peer), stg, kXWarpBytes,
                         peer_of(smem_u32(&bars[bXFull + 8 * pb + warp]), peer));
            bulk_commit();
          }
          // 2. My 16 columns of my quarter: y = scaled S + X (-inf where
          //    masked), kept in TMEM; P against the running maximum of the
          //    earlier tiles into my P units; its row sum; the tile maximum.
          uint32_t mk = 0;  // bit 4e + u: token 32c + 16ch + 4u + e of this sub-tile
          {
            const int shift = 16 * sub + 8 * static_cast<int>(c) + 4 * ch;
#pragma unroll
            for (int e = 0; e < 4; ++e) mk |= ((mkw[e] >> shift) & 0xFu) << (4 * e);
          }
          mbar_wait(&bars[bXFull + 8 * pb + warp], (n_sub >> 1) & 1, abort_flag, p.d_error, kWaitNs);
          // The PV of two sub-tiles back is done: this P buffer is free, and
          // the peer's P of that sub-tile has landed, so this P barrier is
          // in its next phase.  (The quadrant's P copy of that sub-tile was
          // read before the pair barriers of the sub-tile between.)
          if (n_sub >= 2) mbar_wait(&bars[bPvDone + pb], ((n_sub - 2) >> 1) & 1, abort_flag, p.d_error, kWaitNs);
          if (warp == 0 && lane == 0) mbar_expect_tx(&bars[bPIn + pb], kPInBytes);
          const float mm = m == -INFINITY ? 0.f : m;  // all y are -inf when m is
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
          {
            uint32_t v[16];
            tmem_ld16(tSb + 32 * c + 16 * ch, v);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float4 x4 = *reinterpret_cast<const float4*>(sXw + swz<64>(lane * 64 + u * 16));
              const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const bool ok = (mk >> (4 * e + u)) & 1u;
                const float y = ok ? fmaf(__uint_as_float(v[4 * u + e]), p.scale_log2, xs[e]) : -INFINITY;
                mx[e] = fmaxf(mx[e], y);
                v[4 * u + e] = __float_as_uint(y);
              }
            }
            tmem_st16(tSb + 32 * c + 16 * ch, v);
#pragma unroll
            for (int w = 0; w < 2; ++w) {
              float pv[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                pv[e] = ex2_approx(__uint_as_float(v[8 * w + e]) - mm);
                ls[e & 3] += pv[e];
              }
              *reinterpret_cast<uint4*>(sPw + swz<32>(i * 32 + w * 16)) =
                  make_uint4(pack_bf16x2(pv[0], pv[1]), pack_bf16x2(pv[2], pv[3]), pack_bf16x2(pv[4], pv[5]),
                             pack_bf16x2(pv[6], pv[7]));
            }
          }
          const float mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
          tmem_wait_st();
          // 3. Swap tile maxima: this warp's 32 with the peer's same warp; the
          //    quadrant's four per head (two warps, two CTAs) decide alike in
          //    both CTAs and both warps.
          sMaxOut[64 * qd + 32 * ch + lane] = mloc;
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            bulk_to_peer(peer_of(smem_u32(sMaxIn + 64 * qd + 32 * ch), peer), sMaxOut + 64 * qd + 32 * ch, 128,
                         peer_of(smem_u32(&bars[bMaxFull + qd]), peer));
            bulk_commit();
          }
          named_bar_sync(pair_bar, 64);  // the partner warp's maxima are in place
          mbar_wait(&bars[bMaxFull + qd], n_sub & 1, abort_flag, p.d_error, kWaitNs);
          const float mt = fmaxf(fmaxf(sMaxOut[64 * qd + lane], sMaxOut[64 * qd + 32 + lane]),
                                 fmaxf(sMaxIn[64 * qd + lane], sMaxIn[64 * qd + 32 + lane]));
          const bool need = mt > m + kLazy || (m == -INFINITY && mt > -INFINITY);
          float alpha = 1.f;
          if (!__any_sync(0xFFFFFFFFu, need)) {
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
          } else {
            // Rare (a segment's first sub-tile, or a head's maximum grew by
            // more than the lazy threshold): move the running maximum,
            // rescale the row sum (and below, my O columns), and recompute
            // my P units from y.
            if (need) {
              alpha = m == -INFINITY ? 0.f : ex2_approx(m - mt);
              m = mt;
            }
            l *= alpha;
            const float mm2 = m == -INFINITY ? 0.f : m;
            float lr[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t v[16];
            tmem_ld16(tSb + 32 * c + 16 * ch, v);
#pragma unroll
            for (int w = 0; w < 2; ++w) {
              float pv[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                pv[e] = ex2_approx(__uint_as_float(v[8 * w + e]) - mm2);
                lr[e & 3] += pv[e];
              }
              *reinterpret_cast<uint4*>(sPw + swz<32>(i * 32 + w * 16)) =
                  make_uint4(pack_bf16x2(pv[0], pv[1]), pack_bf16x2(pv[2], pv[3]), pack_bf16x2(pv[4], pv[5]),
                             pack_bf16x2(pv[6], pv[7]));
            }
            l += (lr[0] + lr[1]) + (lr[2] + lr[3]);
          }
          // S of this sub-tile has been read for the last time.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[bSUsed + sb]);
          // alpha == 0 only while m was -inf: O then holds zeros (every P so
          // far was 0) or, on a segment's first sub-tile, values that this
          // sub-tile's PV overwrites; either way nothing needs scaling.
          if (__any_sync(0xFFFFFFFFu, alpha != 1.f && alpha != 0.f)) {
            // O must hold the previous sub-tile's PV before it is scaled.
            mbar_wait(&bars[bPvDone + ((n_sub - 1) & 1)], ((n_sub - 1) >> 1) & 1, abort_flag, p.d_error, kWaitNs);
            tc_fence_after();
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
              uint32_t o[16];
              tmem_ld16(tO + 128 * ch + 16 * j, o);
#pragma unroll
              for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st16(tO + 128 * ch + 16 * j, o);
            }
            tmem_wait_st();
          }
          // 4. My P rows (1 KB) to the peer; this warp's wait at the start
          //    of the next sub-tile covers the copy's reads.
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[bPMine2 + pb]);  // the tensor core may start on this CTA's tokens
          __syncwarp();
          if (lane == 0) {
            // The peer's block for these rows is free: the peer's warps
            // waited for their PV of two sub-tiles back (its last reader)
            // before the score pass that preceded the maxima received above.
            uint8_t* blk = sPw + qd * 1024;
            bulk_to_peer(peer_of(smem_u32(blk), peer), blk, kPWarpBytes, peer_of(smem_u32(&bars[bPIn + pb]), peer));
            bulk_commit();
          }
        }
      }

      // The next query token's Q goes into TMEM first (this token's last
      // S = Q K^T has completed: its sub-tile's softmax waited for it), so
      // that the next S runs during this epilogue; O is safe until this
      // warp's next P lets the tensor core start the next O += P V.
      if (seg_end < span.g_end) load_q(qidx + 1);
      // Epilogue of this query token (or split): the row sum over both
      // column halves of both CTAs, added in CTA order so both CTAs agree
      // bit for bit; then my O columns / l.
      const uint32_t sp = n_seg & 1;
      sStatsOut[128 * ch + i] = l;
      fence_proxy_async_smem();
      // Every warp's copies out of the P buffers have been read once all
      // pass this barrier: the O rows below are staged there.
      if (lane == 0) bulk_wait_read();
      named_bar_sync(1, kSoftThreads);
      if (warp == 0 && lane == 0) {
        bulk_to_peer(peer_of(smem_u32(sStats + sp * 256), peer), sStatsOut, 1024,
                     peer_of(smem_u32(&bars[bStatsIn + sp]), peer));
        bulk_commit_and_wait_read();
      }
      mbar_wait(&bars[bStatsIn + sp], (n_seg >> 1) & 1, abort_flag, p.d_error, kWaitNs);
      const float l_mine = sStatsOut[i] + sStatsOut[128 + i];
      const float l_peer = sStats[sp * 256 + i] + sStats[sp * 256 + 128 + i];
      const float lt = c == 0 ? l_mine + l_peer : l_peer + l_mine;
      const float linv = lt > 0.f ? 1.f / lt : 0.f;
      const int nsplit = p.num_splits[qidx + 1] - p.num_splits[qidx];
      const int local = seg_begin == span.g_begin ? span.first_local_split : 0;
      const int64_t split = static_cast<int64_t>(p.num_splits[qidx]) + local;
      const bool direct = nsplit == 1;
      const bool split_ok = direct || (split >= 0 && split < p.ws_splits_cap && local < nsplit);
      if (c == 0 && ch == 0) {
        const float lse = lt > 0.f ? (m + lg2_approx(lt)) * 0.6931471805599453f : -INFINITY;
        const int64_t hrow = static_cast<int64_t>(qidx) * p.h_q + i;
        if (direct)
          p.lse[hrow] = lse;
        else if (split_ok)
          p.ws_lse[split * p.h_q + i] = lse;
        if (!split_ok && p.d_error) atomicOr(p.d_error, MLA_DEVERR_BAD_METADATA);
      }
      m = -INFINITY;
      l = 0.f;
      mbar_wait(&bars[bOReady], n_seg & 1, abort_flag, p.d_error, kWaitNs);
      __syncwarp();
      tc_fence_after();
      // O rows leave through this warp's 4 KB of the P buffers (idle now:
      // every PV of this token is done, and the peer sends its next P only
      // after this CTA's next partial scores): each 32-dim block of the
      // warp's 32 rows is staged there and written by one TMA store.
      uint8_t* ost = sP + warp * 4096;
      // The fused epilogue's records: this lane's head row, bytes d0 .. d0+31
      // and scale byte 512 + d0 / 32 for each 32-dim block d0 of this warp.
      const bool rope = kRope && direct;
      uint8_t* rec = rope ? p.rope_out + (static_cast<int64_t>(qidx) * p.h_q + i) * 528 : nullptr;
      uint32_t sbytes = 0;
      // The warps holding dims 448..511 take pair m's angle once, in lane m,
      // for all 32 rows (it depends on the position and m only).
      float rope_cs = 1.f, rope_sn = 0.f;
      if (rope && static_cast<int>(c) * kHalf + 128 * ch + 96 >= 448)
        rope_cos_sin(static_cast<double>(p.positions[qidx]), p.rope.f[lane], rope_cs, rope_sn);
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        uint32_t o[32];
        tmem_ld32(tO + 128 * ch + 32 * j, o);
        const int d0 = static_cast<int>(c) * kHalf + 128 * ch + 32 * j;
        if constexpr (kRope) {
          if (rope) {
            // O / l, the conjugate rotation of dims 448..511 (pairs
            // (448 + 2m, 449 + 2m)), then E4M3FN under the block's e8m0 scale:
            // the arithmetic of the merge kernel's fused epilogue.
            float v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(o[k]) * linv;
            if (d0 >= 448) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int m = (d0 - 448) / 2 + e;  // lane m holds pair m's angle
                rope_conj_apply(v[2 * e], v[2 * e + 1], __shfl_sync(0xFFFFFFFFu, rope_cs, m),
                                __shfl_sync(0xFFFFFFFFu, rope_sn, m));
              }
            }
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
            const int ex = fp8_block_exponent(amax);
            uint32_t w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              w[u] = e4m3x2(ldexpf(v[4 * u], -ex), ldexpf(v[4 * u + 1], -ex)) |
                     (e4m3x2(ldexpf(v[4 * u + 2], -ex), ldexpf(v[4 * u + 3], -ex)) << 16);
            if (rope_al16) {
              *reinterpret_cast<uint4*>(rec + d0) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4*>(rec + d0 + 16) = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
#pragma unroll
              for (int u = 0; u < 8; ++u) *reinterpret_cast<uint32_t*>(rec + d0 + 4 * u) = w[u];
            }
            sbytes |= static_cast<uint32_t>(127 + ex) << (8 * j);
            __syncwarp();
            continue;
          }
        }
        if (direct) {
          // TMA stores: the 32 x 64-byte block goes out as one tiled store
          // (the staging block's 64-byte swizzle is the tensor map's), from
          // two staging halves in turn.
          uint8_t* st = ost + (j & 1) * 2048;
          if (j >= 2) {
            if (lane == 0) bulk_wait_read_1();  // the store of block j - 2 has read this half
            __syncwarp();
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(st + swz<64>(lane * 64 + u * 16)) =
                make_uint4(pack_bf16x2(__uint_as_float(o[8 * u + 0]) * linv, __uint_as_float(o[8 * u + 1]) * linv),
                           pack_bf16x2(__uint_as_float(o[8 * u + 2]) * linv, __uint_as_float(o[8 * u + 3]) * linv),
                           pack_bf16x2(__uint_as_float(o[8 * u + 4]) * linv, __uint_as_float(o[8 * u + 5]) * linv),
                           pack_bf16x2(__uint_as_float(o[8 * u + 6]) * linv, __uint_as_float(o[8 * u + 7]) * linv));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&out_map, st, d0, qidx * p.h_q + 32 * qd);
            bulk_commit();
          }
        } else if (split_ok) {
          // The same for an fp32 partial: 32 x 128-byte blocks with the
          // 128-byte swizzle, one staging block (4 KB) per warp.
          if (j >= 1) {
            if (lane == 0) bulk_wait_read();
            __syncwarp();
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4*>(ost + swz<128>(lane * 128 + u * 16)) =
                make_float4(__uint_as_float(o[4 * u + 0]) * linv, __uint_as_float(o[4 * u + 1]) * linv,
                            __uint_as_float(o[4 * u + 2]) * linv, __uint_as_float(o[4 * u + 3]) * linv);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&ws_map, ost, d0, static_cast<int>(split) * p.h_q + 32 * qd);
            bulk_commit();
          }
        }
        __syncwarp();  // this warp's staging block is rewritten next
      }
      if constexpr (kRope) {
        if (rope) *reinterpret_cast<uint32_t*>(rec + 512 + 8 * static_cast<int>(c) + 4 * ch) = sbytes;
      }
      // No warp sends the next partial scores (after which the peer's next P
      // lands here) or writes the next P before every warp's O rows have
      // been read out of the P buffers (by the TMA stores too).
      if (lane == 0) bulk_wait_read();
      __syncwarp();
      named_bar_sync(1, kSoftThreads);
      tc_fence_before();
      ++n_seg;
    }
    // This warp's last copies out of shared memory, and the TMA stores'
    // writes, are complete.
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer is done with this CTA's shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


}  // namespace

int decode_pair_smem_bytes() { return PairSmem::kAlloc; }

cudaError_t launch_decode_pair(const DecodeParams& p, int num_parts, cudaStream_t stream) {
  constexpr int smem = PairSmem::kAlloc;
  const bool rope = p.rope_out != nullptr;
  static std::atomic<uint64_t> configured{0}, configured_rope{0};
  cudaError_t e0 = rope ? max_dynamic_smem_once(configured_rope,
                                                reinterpret_cast<const void*>(sparse_decode_pair_kernel<true>), smem)
                        : max_dynamic_smem_once(configured,
                                                reinterpret_cast<const void*>(sparse_decode_pair_kernel<false>), smem);
  if (e0 != cudaSuccess) return e0;
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap kv_map;
  {
    // The FP8 pool as [tokens][528 bytes]; rows gathered 256 bytes (one CTA's half of a record's dims) at a time.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRecFp8), static_cast<cuuint64_t>(p.pool_tokens)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRecFp8)};
    const cuuint32_t estr[2] = {1, 1};
    const cuuint32_t box[2] = {256, 1};
    if (enc(&kv_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.kv), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Outputs and split partials leave by TMA stores: out as [rows][512] bf16,
  // the partials as [rows][512] fp32, in boxes of 32 rows x 32 dims (both
  // buffers are 16-byte aligned, as the entry points check).  A map that is
  // not needed (no bf16 output, no workspace) stays a copy of kv_map.
  CUtensorMap out_map = kv_map, ws_map = kv_map;
  if (p.out != nullptr) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(p.nq) * p.h_q};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&out_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.out, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (p.ws_o != nullptr && p.ws_splits_cap > 0) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(p.ws_splits_cap) * p.h_q};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&ws_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.ws_o, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (rope)
    sparse_decode_pair_kernel<true><<<2 * num_parts, kPThreads, smem, stream>>>(p, kv_map, out_map, ws_map);
  else
    sparse_decode_pair_kernel<false><<<2 * num_parts, kPThreads, smem, stream>>>(p, kv_map, out_map, ws_map);
  return cudaGetLastError();
}

}  // namespace mla
