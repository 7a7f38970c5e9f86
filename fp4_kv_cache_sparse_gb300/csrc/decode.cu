// decode.cu -- token-sparse MLA decode kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes ("flops/flashmla-decode-fp8-fp4-kv", sections "Arithmetic
// intensity" and "Workarounds"; "deepseek-ai/FlashMLA", "How to use it"):
// for each query token and head, attention over the tokens named by the
// indices tensor, each token's 512-dim latent decoded from its FP8 (main
// cache) or FP4 (extra cache) record and used as both key and value, one
// online softmax over all selected tokens, output plus log-sum-exp.
//
// One CTA (384 threads, one per SM) owns one head group (NH heads) of a
// contiguous run of (query token, 128-slot tile) work items:
//   warps 4-11  producers.  Each warp owns 16 token rows of a tile.  Record
//               bytes are loaded with 16-byte read-only loads one whole tile
//               ahead (registers), indices two tiles ahead; a quarter (128
//               dims) is dequantized exactly to bf16 in registers and stored
//               into shared memory in the 128-byte-swizzled canonical layout
//               as soon as the tensor core has released that quarter.
//               Lane 0 of warp 4 also fetches each query token's Q by TMA.
//   warps 0-3   softmax; thread 0 also issues the tensor-core work:
//               S^T = K Q^T (M = 128 tokens, N = NH heads, K = 512) into TMEM
//               quarter by quarter as the producers deliver them, then
//               O^T += V^T P^T (M = 128 dims per quarter, N = NH, K = 128
//               tokens).  The same shared tile is the K-major A operand of
//               the first product and the MN-major A operand of the second.
//               Thread i owns TMEM lane i (token i): it scales and masks its
//               row of S^T and checks it against the running per-head maxima;
//               only when some score exceeds its head's maximum by more than
//               2^8 are exact column maxima computed (shuffle reduce-scatter)
//               and O^T, l rescaled.  P^T goes to shared memory; each thread's
//               running row sums live in spare TMEM columns of its own lane
//               until the end of the query token.
// Hand-offs use mbarriers (tensor-core completion via tcgen05.commit, TMA
// completion via transaction counts) and one named barrier inside the
// softmax warps.  Every mbarrier wait is bounded (see mbar_wait).
#include <cstdint>
#include <cuda.h>

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarps = 8;
constexpr int kRowsPerProducerWarp = kTile / kProducerWarps;  // 16
constexpr int kRounds = kRowsPerProducerWarp / 4;              // 4 loads of 4 tokens x 8 lanes
constexpr uint64_t kWaitLimitNs = 2000000000ull;               // 2 s per wait

// Scores may exceed the running maximum they are exponentiated against by
// up to 2^kLazy before the maximum is moved (P <= 2^8 stays exact enough in
// bf16 and the fp32 sums cannot overflow).
constexpr float kLazyRescale = 8.0f;

template <int NH>
struct Smem {
  static constexpr int kKvBytes = 8 * 128 * 128;        // 8 chunks of 128 tokens x 64 dims (bf16)
  static constexpr int kQBytes = NH * kD * 2;           // NH heads x 512 dims (bf16)
  static constexpr int kPBytes = kTile * NH * 2;        // 128 tokens x NH heads (bf16)
  static constexpr int kKvOff = 0;
  static constexpr int kQOff = kKvOff + kKvBytes;
  static constexpr int kPOff = kQOff + kQBytes;
  static constexpr int kMiscOff = kPOff + kPBytes;
  static constexpr int kBarOff = kMiscOff;              // 16 mbarriers
  static constexpr int kScalarOff = kBarOff + 16 * 8;
  static constexpr int kRedOff = kScalarOff + 64;       // float[4][NH]
  static constexpr int kMOff = kRedOff + 4 * NH * 4;    // float[NH]
  static constexpr int kAlphaOff = kMOff + NH * 4;      // float[NH]
  static constexpr int kLinvOff = kAlphaOff + NH * 4;   // float[NH]
  static constexpr int kEnd = kLinvOff + NH * 4;
  static constexpr int kAlloc = kEnd + 1024;            // + alignment slack
  static constexpr uint32_t kTmemCols = NH == 64 ? 512 : (NH == 32 ? 256 : 128);
};

enum Bar { kQuarterFull = 0, kQuarterFree = 4, kSFull = 8, kOReady, kQFull, kQFree, kDrain };

// Reduce-scatter of v[N] over the 32 lanes of a warp.  Afterwards lane l
// holds in v[0 .. max(N/32,1)) the reduction over all lanes of heads
// rs_head<N>(l, k).  Each step halves the values a lane keeps and exchanges
// the other half with the partner lane.
template <int SIZE, int O>
struct ReduceScatter {
  template <int N, typename Op>
  __device__ __forceinline__ static void run(float (&v)[N], int lane, Op op) {
    if constexpr (O == 0) {
      return;
    } else if constexpr (SIZE == 1) {
      v[0] = op(v[0], __shfl_xor_sync(0xFFFFFFFFu, v[0], O));
      ReduceScatter<1, O / 2>::run(v, lane, op);
    } else {
      constexpr int H = SIZE / 2;
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int k = 0; k < H; ++k) {
        const float send = up ? v[k] : v[k + H];
        const float keep = up ? v[k + H] : v[k];
        v[k] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, send, O));
      }
      ReduceScatter<H, O / 2>::run(v, lane, op);
    }
  }
};

template <int N>
__device__ __forceinline__ int rs_head(int lane, int k) {
  if constexpr (N >= 32)
    return (N / 32) * lane + k;
  else
    return lane / (32 / N);
}

struct MaxOp {
  __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct AddOp {
  __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Record bytes: read once, so not kept in L1; the L2 fetches the 256-byte
// block around each piece, which holds the neighbouring pieces of the same
// record that later quarters read (a 128-byte quarter slice straddles lines).
__device__ __forceinline__ uint4 ldg_stream16(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream8(const uint8_t* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ldg_u4(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u32(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u8(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// TMA: arm an mbarrier with the bytes it will receive; 2-D tiled load.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// One elected lane of a converged warp issues: D[tmem] (+)= A[smem] * B[smem].
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
// (asynchronous work already issued must complete before TMEM and shared
// memory go away) but gives up after its own limit.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, int32_t* d_error) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63) == 63 && global_timer_ns() - t0 > kWaitLimitNs) {
      if (d_error) atomicOr(d_error, MLA_DEVERR_TIMEOUT);
      return;
    }
  }
}

// Work decomposition shared by all roles of a CTA.
struct Span {
  int64_t g_begin, g_end;
  int first_local_split;
  bool ok;
};

__device__ __forceinline__ Span load_span(const DecodeParams& p, int part) {
  Span s;
  const int32_t* e = p.sched + static_cast<int64_t>(part) * MLA_SCHED_INTS;
  s.g_begin = e[0];
  s.g_end = e[1];
  s.first_local_split = e[2];
  const int64_t G = static_cast<int64_t>(p.nq) * p.T;
  s.ok = s.g_begin >= 0 && s.g_begin <= s.g_end && s.g_end <= G && s.first_local_split >= 0;
  if (!s.ok) s.g_begin = s.g_end = 0;
  return s;
}

// Index-slot geometry of tile t of a query token.
struct TileInfo {
  const int32_t* ids;   // row of the indices tensor this tile reads
  int slot0;            // first slot of the tile within that row
  int nslots;           // row length (topk or extra_topk)
  bool extra;           // FP4 extra cache
  int64_t pool;         // tokens in the pool the tile reads
};

__device__ __forceinline__ TileInfo tile_info(const DecodeParams& p, int qidx, int t) {
  TileInfo ti;
  if (t < p.Tm) {
    ti.ids = p.idx + static_cast<int64_t>(qidx) * p.topk;
    ti.slot0 = t * kTile;
    ti.nslots = p.topk;
    ti.extra = false;
    ti.pool = p.pool_tokens;
  } else {
    ti.ids = p.xidx + static_cast<int64_t>(qidx) * p.xtopk;
    ti.slot0 = (t - p.Tm) * kTile;
    ti.nslots = p.xtopk;
    ti.extra = true;
    ti.pool = p.xpool_tokens;
  }
  return ti;
}

// One producer lane's view of a tile: the raw index of its token in each
// load round (-1 past the end of the row), fetched two tiles ahead and only
// checked against the pool when its bytes are requested, one tile later, so
// that the index loads' latency stays hidden.
struct LaneTile {
  int32_t id[kRounds];
  bool extra;
};

__device__ __forceinline__ LaneTile lane_tile(const DecodeParams& p, int g, int row0) {
  LaneTile lt;
  // Items number fewer than 2^31 (the host checks), so 32-bit division.
  const int qidx = g / p.T;
  const TileInfo ti = tile_info(p, qidx, g - qidx * p.T);
  lt.extra = ti.extra;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int slot = ti.slot0 + row0 + r * 4;
    lt.id[r] = slot < ti.nslots ? __ldg(ti.ids + slot) : -1;
  }
  return lt;
}

// Entries outside [0, pool) become -1 (skipped); all but -1 are flagged.
__device__ __forceinline__ void validate(const DecodeParams& p, LaneTile& lt, bool flag_bad) {
  const int64_t pool = lt.extra ? p.xpool_tokens : p.pool_tokens;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int32_t id = lt.id[r];
    const bool valid = id >= 0 && static_cast<int64_t>(id) < pool;
    if (!valid && id != -1 && flag_bad && p.d_error) atomicOr(p.d_error, MLA_DEVERR_BAD_INDEX);
    lt.id[r] = valid ? id : -1;
  }
}

// Register-resident bytes of one quarter (128 dims) of the lane's 4 tokens.
struct QuarterRegs {
  uint4 data[kRounds];   // FP8: 16 e4m3 bytes; FP4: .x/.y = 8 bytes of e2m1 pairs
  uint32_t scale[kRounds];
};

// seg = 16-dim segment of the lane within the quarter (0..7): dims
// 128 qq + 16 seg .. +15.  kFp8Scale: the quarter's FP8 scale word is loaded
// here (otherwise load_scales_fp8 loads all four quarters' at once).
template <bool kFp8Scale>
__device__ __forceinline__ void load_quarter(const DecodeParams& p, const LaneTile& lt, int qq, int seg,
                                             QuarterRegs& q) {
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int32_t id = lt.id[r];
    if (id < 0) {
      q.data[r] = make_uint4(0, 0, 0, 0);
      q.scale[r] = lt.extra ? 0x38u : 127u * 0x01010101u;
    } else if (!lt.extra) {
      const uint8_t* rec = p.kv + static_cast<int64_t>(id) * kRecFp8;
      q.data[r] = ldg_stream16(rec + qq * 128 + seg * 16);
      if constexpr (kFp8Scale) q.scale[r] = ldg_u32(rec + 512 + qq * 4);
    } else {
      const uint8_t* rec = p.xkv + static_cast<int64_t>(id) * kRecFp4;
      const uint2 d = ldg_stream8(rec + qq * 64 + seg * 8);
      q.data[r] = make_uint4(d.x, d.y, 0, 0);
      q.scale[r] = ldg_u8(rec + 256 + qq * 8 + seg);
    }
  }
}

// FP8 tiles: the 16 scale bytes of each of the lane's rows in one load; word
// qq goes to quarter qq's registers.  Called once the current tile's last
// quarter has been stored (every quarter's scale registers are free then).
// With 64 heads this replaces four 4-byte loads per row (fp8_b64_h64 80.9 ->
// 76.9 us); with 16 heads the next tile's first quarter follows too soon
// for loads issued this late (long_dense_b32_h16 482 -> 526 us), so fewer
// heads keep the per-quarter loads.
__device__ __forceinline__ void load_scales_fp8(const DecodeParams& p, const LaneTile& lt, QuarterRegs (&buf)[4]) {
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int32_t id = lt.id[r];
    const uint4 s = id >= 0 ? ldg_u4(p.kv + static_cast<int64_t>(id) * kRecFp8 + 512)
                            : make_uint4(127u * 0x01010101u, 127u * 0x01010101u, 127u * 0x01010101u,
                                         127u * 0x01010101u);
    buf[0].scale[r] = s.x;
    buf[1].scale[r] = s.y;
    buf[2].scale[r] = s.z;
    buf[3].scale[r] = s.w;
  }
}

// kRope: query tokens of one split leave as FP8 records after the
// conjugate rotary embedding (the fused epilogue) instead of bf16 rows; a
// separate instantiation, so that the bf16 kernel carries none of it.
template <int NH, bool kRope>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap q_map) {
  using L = Smem<NH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKV = smem + L::kKvOff;
  uint8_t* sQ = smem + L::kQOff;
  uint8_t* sP = smem + L::kPOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kScalarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kScalarOff + 4);
  float* red = reinterpret_cast<float*>(smem + L::kRedOff);
  float* sm_m = reinterpret_cast<float*>(smem + L::kMOff);
  float* sm_alpha = reinterpret_cast<float*>(smem + L::kAlphaOff);
  float* sm_linv = reinterpret_cast<float*>(smem + L::kLinvOff);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int part = blockIdx.x / p.n_hg;
  const int hg = blockIdx.x % p.n_hg;

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kQuarterFull + i], kProducerWarps);
      mbar_init(&bars[kQuarterFree + i], 1);
    }
    mbar_init(&bars[kSFull], 1);
    mbar_init(&bars[kOReady], 1);
    mbar_init(&bars[kQFull], 1);
    mbar_init(&bars[kQFree], 1);
    mbar_init(&bars[kDrain], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (tid < NH) sm_m[tid] = -INFINITY;
  if (warp == 1) tmem_alloc(tmem_slot, L::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const Span span = load_span(p, part);
  if (!span.ok && tid == 0 && p.d_error) atomicOr(p.d_error, MLA_DEVERR_BAD_METADATA);

  if (warp >= 4) {
    // ------------------------------------------------------------------
    // Producers.
    // ------------------------------------------------------------------
    const int pw = warp - 4;
    // Lane geometry: lane = c1 * 16 + t4 * 4 + s4.  A load instruction
    // covers 4 tokens (t4) x 2 chunks of the quarter (c1) x 4 16-byte
    // segments (s4); a store phase (8 consecutive lanes) covers two adjacent
    // rows, whose different swizzle patterns put the 8 stores in 8 different
    // bank groups.
    const int s4 = lane & 3;
    const int t4 = (lane >> 2) & 3;
    const int c1 = lane >> 4;
    const int seg = c1 * 4 + s4;        // 16-dim segment within the quarter
    const int row0 = pw * kRowsPerProducerWarp + t4;
    const bool flag_bad = hg == 0 && seg == 0;
    // Byte offsets of the lane's two 16-byte units in its chunk for row
    // row0 + 4 r: the row's low 3 bits are t4 + 4 (r & 1).
    uint32_t off_even[2], off_odd[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const uint32_t row = row0 + 4 * rr;
      off_even[rr] = swz<128>(row * 128 + (2 * s4) * 16);
      off_odd[rr] = swz<128>(row * 128 + (2 * s4 + 1) * 16);
    }
    const int sshift = 8 * (2 * c1 + (s4 >> 1));  // scale byte within the quarter's scale word
    constexpr bool kScalePerQuarter = NH < 64;

    uint32_t n_tile = 0, n_seg = 0;
    int64_t g = span.g_begin;
    LaneTile cur{}, nxt{};
    QuarterRegs buf[4];
    if (g < span.g_end) {
      cur = lane_tile(p, static_cast<int>(g), row0);
      validate(p, cur, flag_bad);
      if (g + 1 < span.g_end) nxt = lane_tile(p, static_cast<int>(g + 1), row0);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) load_quarter<kScalePerQuarter>(p, cur, qq, seg, buf[qq]);
      if (!kScalePerQuarter && !cur.extra) load_scales_fp8(p, cur, buf);
    }
    int64_t seg_end = g;  // forces a segment start on the first tile
    for (; g < span.g_end; ++g, ++n_tile) {
      if (g == seg_end) {
        // First tile of a query token: its Q by TMA once the previous
        // token's last S^T no longer reads shared Q.
        const int qidx = static_cast<int>(g / p.T);
        seg_end = min(span.g_end, static_cast<int64_t>(qidx + 1) * p.T);
        if (pw == 0 && lane == 0) {
          if (n_seg > 0) mbar_wait(&bars[kQFree], (n_seg - 1) & 1, abort_flag, p.d_error, kWaitLimitNs);
          mbar_expect_tx(&bars[kQFull], NH * kD * 2);
          const int y = qidx * p.h_q + hg * NH;
#pragma unroll
          for (int c = 0; c < 8; ++c) tma_load_2d(sQ + c * (NH * 128), &q_map, c * 64, y, &bars[kQFull]);
        }
        ++n_seg;
      }
      const bool extra = cur.extra;
      LaneTile nxt2{};
      if (g + 2 < span.g_end) nxt2 = lane_tile(p, static_cast<int>(g + 2), row0);
      if (g + 1 < span.g_end) validate(p, nxt, flag_bad);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        if (n_tile > 0) mbar_wait(&bars[kQuarterFree + qq], (n_tile - 1) & 1, abort_flag, p.d_error, kWaitLimitNs);
        uint8_t* chunk = sKV + (2 * qq + c1) * 16384;
        if (!extra) {
          uint32_t sb[kRounds];
          bool big = false;
#pragma unroll
          for (int r = 0; r < kRounds; ++r) {
            sb[r] = (buf[qq].scale[r] >> sshift) & 0xFFu;
            big |= sb[r] > 142u;
          }
          const bool any_big = __any_sync(0xFFFFFFFFu, big);
#pragma unroll
          for (int r = 0; r < kRounds; ++r) {
            uint32_t o[8];
            if (!any_big)
              dequant_fp8_16_small_scale(buf[qq].data[r], sb[r], o);
            else
              dequant_fp8_16(buf[qq].data[r], sb[r], o);
            const uint32_t radd = (r >> 1) * 1024;  // rows r and r + 2 differ by 8 rows
            *reinterpret_cast<uint4*>(chunk + off_even[r & 1] + radd) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(chunk + off_odd[r & 1] + radd) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        } else {
#pragma unroll
          for (int r = 0; r < kRounds; ++r) {
            uint32_t o[8];
            dequant_fp4_16(buf[qq].data[r].x, buf[qq].data[r].y, buf[qq].scale[r], o);
            const uint32_t radd = (r >> 1) * 1024;
            *reinterpret_cast<uint4*>(chunk + off_even[r & 1] + radd) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(chunk + off_odd[r & 1] + radd) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kQuarterFull + qq]);
        // The registers of this quarter now take the next tile's bytes.
        if (g + 1 < span.g_end) {
          if (!kScalePerQuarter && qq == 3 && !nxt.extra) load_scales_fp8(p, nxt, buf);
          load_quarter<kScalePerQuarter>(p, nxt, qq, seg, buf[qq]);
        }
      }
      cur = nxt;
      nxt = nxt2;
    }
  } else {
    // ------------------------------------------------------------------
    // Softmax (+ tensor-core issue by thread 0) and epilogue.
    // ------------------------------------------------------------------
    const int i = tid;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // TMEM columns: S^T [0, NH), O^T quarters [NH, 5 NH), row sums [5 NH, 6 NH).
    const uint32_t tS = tmem + lane_base, tO = tmem + lane_base + NH, tL = tmem + lane_base + 5 * NH;
    constexpr int V = NH >= 32 ? NH / 32 : 1;  // values a lane keeps after a reduce-scatter
    constexpr uint32_t idesc_qk = make_idesc_bf16(128, NH, false, false);
    constexpr uint32_t idesc_pv = make_idesc_bf16(128, NH, true, true);
    constexpr uint32_t p_sbo = 8 * 2 * NH;        // 8 rows of P^T
    constexpr uint32_t p_swz = NH == 64 ? kSwizzle128 : (NH == 32 ? kSwizzle64 : kSwizzle32);
    const uint32_t kv_base = smem_u32(sKV), q_base = smem_u32(sQ), p_base = smem_u32(sP);
    uint32_t n_tile = 0, n_seg = 0;
    bool issued = false;
    for (int64_t g = span.g_begin; g < span.g_end;) {
      const int qidx = static_cast<int>(g / p.T);
      const int64_t seg_end = min(span.g_end, static_cast<int64_t>(qidx + 1) * p.T);
      const int64_t seg_begin = g;
      {
        uint32_t z[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) z[k] = 0u;
#pragma unroll
        for (int c = 0; c < NH / 16; ++c) tmem_st16(tL + c * 16, z);
        tmem_wait_st();
      }
      for (; g < seg_end; ++g, ++n_tile) {
        const bool first = g == seg_begin;
        const int t = static_cast<int>(g - static_cast<int64_t>(qidx) * p.T);
        const TileInfo ti = tile_info(p, qidx, t);
        const int slot = ti.slot0 + i;
        const int32_t id = slot < ti.nslots ? __ldg(ti.ids + slot) : -1;
        const bool valid = id >= 0 && static_cast<int64_t>(id) < ti.pool;

        if (warp == 0) {
          // S^T = K Q^T over the 8 dim chunks, as quarters arrive (the whole
          // warp waits; one elected lane issues).
          if (first) mbar_wait(&bars[kQFull], n_seg & 1, abort_flag, p.d_error, kWaitLimitNs);
#pragma unroll 1
          for (int qq = 0; qq < 4; ++qq) {
            mbar_wait(&bars[kQuarterFull + qq], n_tile & 1, abort_flag, p.d_error, kWaitLimitNs);
            __syncwarp();
            tc_fence_after();
            // First K step's descriptors; later steps only move the start
            // address (the 14-bit field cannot carry below 256 KB).
            const uint64_t a0 = make_smem_desc(kv_base + 2 * qq * 16384, 16, 1024, kSwizzle128);
            const uint64_t b0 = make_smem_desc(q_base + 2 * qq * (NH * 128), 16, 1024, kSwizzle128);
#pragma unroll 2
            for (int j = 0; j < 8; ++j)
              mma_ss_elect(tmem, a0 + (((j >> 2) * 16384 + (j & 3) * 32) >> 4),
                           b0 + (((j >> 2) * NH * 128 + (j & 3) * 32) >> 4), idesc_qk, (qq | j) != 0);
          }
          issued = true;
          commit_elect(&bars[kSFull]);
          if (g + 1 == seg_end) commit_elect(&bars[kQFree]);
        }
        mbar_wait(&bars[kSFull], n_tile & 1, abort_flag, p.d_error, kWaitLimitNs);
        __syncwarp();
        tc_fence_after();

        // Pass 1: largest excess of a score over its head's running max.
        float excess = -INFINITY;
#pragma unroll
        for (int c = 0; c < NH / 16; ++c) {
          uint32_t r[16];
          tmem_ld16(tS + c * 16, r);
          const float4* m4 = reinterpret_cast<const float4*>(sm_m + c * 16);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 m = m4[k4];
            excess = fmaxf(excess, __uint_as_float(r[4 * k4 + 0]) * p.scale_log2 - m.x);
            excess = fmaxf(excess, __uint_as_float(r[4 * k4 + 1]) * p.scale_log2 - m.y);
            excess = fmaxf(excess, __uint_as_float(r[4 * k4 + 2]) * p.scale_log2 - m.z);
            excess = fmaxf(excess, __uint_as_float(r[4 * k4 + 3]) * p.scale_log2 - m.w);
          }
        }
        int move_max;
        {
          const int mine = valid && excess > kLazyRescale;
          asm volatile(
              "{\n\t.reg .pred pi, po;\n\t"
              "setp.ne.s32 pi, %1, 0;\n\t"
              "bar.red.or.pred po, 2, %2, pi;\n\t"
              "selp.s32 %0, 1, 0, po;\n\t}"
              : "=r"(move_max)
              : "r"(mine), "r"(kSoftmaxThreads)
              : "memory");
        }
        if (move_max) {
          // Exact column maxima of this tile, 16 heads at a time.
#pragma unroll
          for (int c = 0; c < NH / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(tS + c * 16, r);
            float v[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = valid ? __uint_as_float(r[k]) * p.scale_log2 : -INFINITY;
            ReduceScatter<16, 16>::run(v, lane, MaxOp());
            if ((lane & 1) == 0) red[warp * NH + c * 16 + (lane >> 1)] = v[0];
          }
          named_bar_sync(1, kSoftmaxThreads);
          int any_rescale = 0;
          if (i < NH) {
            const float mt = fmaxf(fmaxf(red[i], red[NH + i]), fmaxf(red[2 * NH + i], red[3 * NH + i]));
            const float m_old = sm_m[i];
            float alpha = 1.f;
            if (mt > m_old + kLazyRescale || (m_old == -INFINITY && mt > -INFINITY)) {
              alpha = m_old == -INFINITY ? 0.f : ex2_approx(m_old - mt);
              any_rescale = m_old != -INFINITY;
              sm_m[i] = mt;
            }
            sm_alpha[i] = alpha;
          }
          asm volatile(
              "{\n\t.reg .pred pi, po;\n\t"
              "setp.ne.s32 pi, %1, 0;\n\t"
              "bar.red.or.pred po, 2, %2, pi;\n\t"
              "selp.s32 %0, 1, 0, po;\n\t}"
              : "=r"(any_rescale)
              : "r"(any_rescale), "r"(kSoftmaxThreads)
              : "memory");
          if (any_rescale) {
#pragma unroll 1
            for (int c = 0; c < NH / 16; ++c) {
              uint32_t o[16];
              tmem_ld16(tL + c * 16, o);
#pragma unroll
              for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * sm_alpha[c * 16 + k]);
              tmem_st16(tL + c * 16, o);
            }
            tmem_wait_st();
            if (!first) {
              // O^T[d, h] *= alpha[h]; the products so far are complete (the
              // tensor core finished them before this tile's S^T).
#pragma unroll 1
              for (int r = 0; r < 4; ++r) {
#pragma unroll
                for (int c = 0; c < NH / 16; ++c) {
                  uint32_t o[16];
                  tmem_ld16(tO + r * NH + c * 16, o);
#pragma unroll
                  for (int k = 0; k < 16; ++k)
                    o[k] = __float_as_uint(__uint_as_float(o[k]) * sm_alpha[c * 16 + k]);
                  tmem_st16(tO + r * NH + c * 16, o);
                }
              }
              tmem_wait_st();
            }
          }
        }
        // Pass 2: P = 2^(x - m), row i of P^T (MN-major, swizzled), row sums.
#pragma unroll 1
        for (int c = 0; c < NH / 16; ++c) {
          uint32_t r[16];
          tmem_ld16(tS + c * 16, r);
          uint32_t l[16];
          tmem_ld16(tL + c * 16, l);
          float pv[16];
          const float4* m4 = reinterpret_cast<const float4*>(sm_m + c * 16);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 m = m4[k4];
            const float mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int k = 4 * k4 + j;
              const float xv = __uint_as_float(r[k]) * p.scale_log2 - mm[j];
              pv[k] = (valid && mm[j] != -INFINITY) ? ex2_approx(xv) : 0.f;
              l[k] = __float_as_uint(__uint_as_float(l[k]) + pv[k]);
            }
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint4 w;
            w.x = pack_bf16x2(pv[8 * u + 0], pv[8 * u + 1]);
            w.y = pack_bf16x2(pv[8 * u + 2], pv[8 * u + 3]);
            w.z = pack_bf16x2(pv[8 * u + 4], pv[8 * u + 5]);
            w.w = pack_bf16x2(pv[8 * u + 6], pv[8 * u + 7]);
            *reinterpret_cast<uint4*>(sP + swz<2 * NH>(i * (2 * NH) + (2 * c + u) * 16)) = w;
          }
          tmem_st16(tL + c * 16, l);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, kSoftmaxThreads);
        if (warp == 0) {
          // O^T += V^T P^T (whole warp; one elected lane issues).
          tc_fence_after();
          const uint64_t pb0 = make_smem_desc(p_base, 16 * p_sbo, p_sbo, p_swz);
#pragma unroll 1
          for (int r = 0; r < 4; ++r) {
            const uint64_t a0 = make_smem_desc(kv_base + 2 * r * 16384, 16384, 1024, kSwizzle128);
#pragma unroll 2
            for (int ks = 0; ks < 8; ++ks)
              mma_ss_elect(tmem + NH + r * NH, a0 + ((ks * 2048) >> 4), pb0 + ((ks * 2 * p_sbo) >> 4), idesc_pv,
                           !(first && ks == 0));
            commit_elect(&bars[kQuarterFree + r]);
          }
          if (g + 1 == seg_end) commit_elect(&bars[kOReady]);
        }
      }

      // Epilogue of this query token (or of this split of it).
      // Column sums of the per-thread row sums.
      {
        float lw[NH];
#pragma unroll
        for (int c = 0; c < NH / 16; ++c) {
          uint32_t l[16];
          tmem_ld16(tL + c * 16, l);
#pragma unroll
          for (int k = 0; k < 16; ++k) lw[c * 16 + k] = __uint_as_float(l[k]);
        }
        ReduceScatter<NH, 16>::run(lw, lane, AddOp());
#pragma unroll
        for (int k = 0; k < V; ++k) {
          if (NH >= 32 || (lane & 1) == 0) red[warp * NH + rs_head<NH>(lane, k)] = lw[k];
        }
      }
      mbar_wait(&bars[kOReady], n_seg & 1, abort_flag, p.d_error, kWaitLimitNs);
      __syncwarp();
      tc_fence_after();
      named_bar_sync(1, kSoftmaxThreads);
      const int nsplit = p.num_splits[qidx + 1] - p.num_splits[qidx];
      const int local = seg_begin == span.g_begin ? span.first_local_split : 0;
      const int64_t split = static_cast<int64_t>(p.num_splits[qidx]) + local;
      const bool direct = nsplit == 1;
      const bool split_ok = direct || (split >= 0 && split < p.ws_splits_cap && local < nsplit);
      if (i < NH) {
        const float l = red[i] + red[NH + i] + red[2 * NH + i] + red[3 * NH + i];
        const float m = sm_m[i];
        sm_linv[i] = l > 0.f ? 1.f / l : 0.f;
        const float lse = l > 0.f ? (m + lg2_approx(l)) * 0.6931471805599453f : -INFINITY;
        const int64_t hrow = static_cast<int64_t>(qidx) * p.h_q + hg * NH + i;
        if (direct)
          p.lse[hrow] = lse;
        else if (split_ok)
          p.ws_lse[split * p.h_q + hg * NH + i] = lse;
        sm_m[i] = -INFINITY;  // reset for the next query token
      }
      if (!split_ok && i == 0 && p.d_error) atomicOr(p.d_error, MLA_DEVERR_BAD_METADATA);
      named_bar_sync(1, kSoftmaxThreads);
      if constexpr (kRope) {
        if (direct) {
          // The fused epilogue's records: dim d of every head's row.  The
          // 32 lanes of a warp hold one 32-dim block (its e8m0 scale is the
          // warp's maximum); dims 448..511 (quarter 3, warps 2 and 3) pair
          // even and odd lanes for the conjugate rotation, each pair's angle
          // taken once per lane pair.  The arithmetic of the merge kernel's
          // fused epilogue, so the bytes agree.
#pragma unroll 1
          for (int r = 0; r < 4; ++r) {
            const int d = r * 128 + i;
            const bool rot = d >= 448;  // uniform in the warp
            float cs = 1.f, sn = 0.f;
            if (rot) rope_cos_sin(static_cast<double>(p.positions[qidx]), p.rope.f[(d - 448) >> 1], cs, sn);
#pragma unroll 1
            for (int c = 0; c < NH / 16; ++c) {
              uint32_t o[16];
              tmem_ld16(tO + r * NH + c * 16, o);
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                const int h = c * 16 + k;
                float v = __uint_as_float(o[k]) * sm_linv[h];
                if (rot) {
                  const float w = __shfl_xor_sync(0xFFFFFFFFu, v, 1);
                  float a = (lane & 1) ? w : v, b = (lane & 1) ? v : w;
                  rope_conj_apply(a, b, cs, sn);
                  v = (lane & 1) ? b : a;
                }
                float amax = fabsf(v);
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o2));
                const int ex = fp8_block_exponent(amax);
                uint8_t* rec = p.rope_out + (static_cast<int64_t>(qidx) * p.h_q + hg * NH + h) * 528;
                rec[d] = static_cast<uint8_t>(e4m3x2(ldexpf(v, -ex), 0.f) & 0xFFu);
                if (lane == 0) rec[512 + (d >> 5)] = static_cast<uint8_t>(127 + ex);
              }
            }
          }
          tc_fence_before();
          named_bar_sync(1, kSoftmaxThreads);  // O and sm_m reads done before the next token's tiles
          ++n_seg;
          continue;
        }
      }
#pragma unroll 1
      for (int r = 0; r < 4; ++r) {
        const int d = r * 128 + i;
#pragma unroll
        for (int c = 0; c < NH / 16; ++c) {
          uint32_t o[16];
          tmem_ld16(tO + r * NH + c * 16, o);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int h = c * 16 + k;
            const float v = __uint_as_float(o[k]) * sm_linv[h];
            if (direct) {
              const int64_t row = static_cast<int64_t>(qidx) * p.h_q + hg * NH + h;
              p.out[row * kD + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
            } else if (split_ok) {
              p.ws_o[(split * p.h_q + hg * NH + h) * kD + d] = v;
            }
          }
        }
      }
      tc_fence_before();
      named_bar_sync(1, kSoftmaxThreads);  // O and sm_m reads done before the next token's tiles
      ++n_seg;
    }
    if (warp == 0 && issued) {
      // Normal runs have completed every product already (the epilogue
      // waited for it); after a timeout this keeps TMEM alive until the
      // tensor core is done with it (the wait ignores the abort flag and
      // has its own bound).
      commit_elect(&bars[kDrain]);
      __syncwarp();
      mbar_wait_drain(&bars[kDrain], 0, p.d_error);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}


}  // namespace

template <int NH>
cudaError_t launch_decode(const DecodeParams& p, int grid, cudaStream_t stream) {
  constexpr int smem = Smem<NH>::kAlloc;
  const bool rope = p.rope_out != nullptr;
  static std::atomic<uint64_t> configured{0}, configured_rope{0};
  cudaError_t e0 =
      rope ? max_dynamic_smem_once(configured_rope, reinterpret_cast<const void*>(sparse_decode_kernel<NH, true>), smem)
           : max_dynamic_smem_once(configured, reinterpret_cast<const void*>(sparse_decode_kernel<NH, false>), smem);
  if (e0 != cudaSuccess) return e0;
  // Q viewed as [nq * h_q rows][512 bf16]; a box is NH rows x 64 dims, 128-byte swizzled.
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap q_map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(p.nq) * p.h_q};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(NH)};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.q), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (rope)
    sparse_decode_kernel<NH, true><<<grid, kThreads, smem, stream>>>(p, q_map);
  else
    sparse_decode_kernel<NH, false><<<grid, kThreads, smem, stream>>>(p, q_map);
  return cudaGetLastError();
}

template cudaError_t launch_decode<16>(const DecodeParams&, int, cudaStream_t);
template cudaError_t launch_decode<32>(const DecodeParams&, int, cudaStream_t);
template cudaError_t launch_decode<64>(const DecodeParams&, int, cudaStream_t);

int decode_smem_bytes(int nh) {
  return nh == 64 ? Smem<64>::kAlloc : (nh == 32 ? Smem<32>::kAlloc : Smem<16>::kAlloc);
}

}  // namespace mla
