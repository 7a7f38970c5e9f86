// decode.cu -- token-sparse MLA decode kernel for sm_103a (tcgen05 + TMEM).
//
// What it computes ("flops/flashmla-decode-fp8-fp4-kv", sections "Arithmetic
// intensity" and "Workarounds"; "deepseek-ai/FlashMLA", "How to use it"):
// for each query token and head, attention over the tokens named by the
// indices tensor, each token's 512-dim latent decoded from its FP8 (main
// cache) or FP4 (extra cache) record and used as both key and value, one
// online softmax over all selected tokens, output plus log-sum-exp.
//
// Structure of one CTA (288 threads), which owns one head group (NH heads)
// of a contiguous run of (query token, tile) work items:
//   warps 4-7  producers: gather the 128 records of a tile with 16-byte
//              read-only loads, dequantize in registers (exact, bf16), write
//              the bf16 tile into shared memory in the 128-byte-swizzled
//              canonical layout, one 128-dim quarter at a time.
//   warp 8     tensor-core issuer: S^T = K Q^T (M = 128 tokens, N = NH heads,
//              K = 512) into TMEM, then O^T += V^T P^T (M = 128 dims per
//              quarter, N = NH, K = 128 tokens).  The same shared tile is the
//              K-major A operand of the first product and the MN-major A
//              operand of the second (K = V = the latent).
//   warps 0-3  softmax: thread i owns TMEM lane i (token i of the tile):
//              scale, mask, column max and sum over the 128 tokens
//              (shuffle reduce-scatter + shared memory), lazy rescale of O,
//              P^T to shared memory; at the end of a query token, normalise
//              O^T and write the output (or a split partial) and the LSE.
// Hand-offs use mbarriers; tensor-core completion is signalled with
// tcgen05.commit.  Every wait is bounded (see mbar_wait).
#include <cstdint>

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kThreads = 288;
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerBase = 128;
constexpr int kMmaWarp = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

// Softmax stays exact with a stale running max as long as the scores it
// subtracts from stay within 2^kLazy of it.
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
  // misc: 16 mbarriers, then scalars, then per-head arrays
  static constexpr int kBarOff = kMiscOff;
  static constexpr int kScalarOff = kBarOff + 16 * 8;
  static constexpr int kRedOff = kScalarOff + 64;       // float[4][NH]
  static constexpr int kMOff = kRedOff + 4 * NH * 4;    // float[NH]
  static constexpr int kAlphaOff = kMOff + NH * 4;      // float[NH]
  static constexpr int kLinvOff = kAlphaOff + NH * 4;   // float[NH]
  static constexpr int kEnd = kLinvOff + NH * 4;
  static constexpr int kAlloc = kEnd + 1024;            // + alignment slack
  static constexpr uint32_t kTmemCols = NH == 64 ? 512 : (NH == 32 ? 256 : 128);
};

enum Bar { kQuarterFull = 0, kQuarterFree = 4, kSFull = 8, kPFull, kOReady, kQFull, kQFree, kDrain };

// Reduce-scatter of v[N] over the 32 lanes of a warp.  Afterwards lane l
// holds in v[0 .. max(N/32,1)) the reduction over all lanes of heads
// head_of(l, k) (see below).  Each step halves the values a lane keeps and
// exchanges the other half with the partner lane.
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

template <int NH>
__global__ void __launch_bounds__(kThreads, 1) sparse_decode_kernel(const DecodeParams p) {
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
      mbar_init(&bars[kQuarterFull + i], 4);
      mbar_init(&bars[kQuarterFree + i], 1);
    }
    mbar_init(&bars[kSFull], 1);
    mbar_init(&bars[kPFull], kSoftmaxThreads);
    mbar_init(&bars[kOReady], 1);
    mbar_init(&bars[kQFull], 4);
    mbar_init(&bars[kQFree], 1);
    mbar_init(&bars[kDrain], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, L::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const Span span = load_span(p, part);
  if (!span.ok && tid == 0 && p.d_error) atomicOr(p.d_error, MLA_DEVERR_BAD_METADATA);

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------
    // Producers: Q of each query token, then the dequantized tiles.
    // ------------------------------------------------------------------
    const int pt = tid - kProducerBase;
    const int pw = pt >> 5;
    const int j4 = lane >> 3;  // token of the 4 a load instruction covers
    const int s8 = lane & 7;   // 16-value segment within a 128-dim quarter
    uint32_t n_tile = 0, n_seg = 0;
    for (int64_t g = span.g_begin; g < span.g_end;) {
      const int qidx = static_cast<int>(g / p.T);
      const int64_t seg_end = min(span.g_end, static_cast<int64_t>(qidx + 1) * p.T);
      // Q (NH heads of this head group), K-major, 128-byte swizzle.
      if (n_seg > 0) mbar_wait(&bars[kQFree], (n_seg - 1) & 1, abort_flag, p.d_error, kWaitLimitNs);
      {
        const uint4* qsrc = reinterpret_cast<const uint4*>(
            p.q + (static_cast<int64_t>(qidx) * p.h_q + static_cast<int64_t>(hg) * NH) * kD);
#pragma unroll 4
        for (int u = pt; u < NH * 64; u += 128) {
          const int h = u >> 6, d8 = u & 63;
          const uint4 v = __ldg(qsrc + u);
          const uint32_t off = (d8 >> 3) * (NH * 128) + swz<128>(h * 128 + (d8 & 7) * 16);
          *reinterpret_cast<uint4*>(sQ + off) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kQFull]);
      }
      for (; g < seg_end; ++g, ++n_tile) {
        const int t = static_cast<int>(g - static_cast<int64_t>(qidx) * p.T);
        const TileInfo ti = tile_info(p, qidx, t);
        const uint8_t* rec[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int slot = ti.slot0 + pw * 32 + r * 4 + j4;
          const int32_t id = slot < ti.nslots ? __ldg(ti.ids + slot) : -1;
          const bool valid = id >= 0 && static_cast<int64_t>(id) < ti.pool;
          if (!valid && id != -1 && hg == 0 && s8 == 0 && p.d_error) atomicOr(p.d_error, MLA_DEVERR_BAD_INDEX);
          rec[r] = !valid ? nullptr
                          : (ti.extra ? p.xkv + static_cast<int64_t>(id) * kRecFp4
                                      : p.kv + static_cast<int64_t>(id) * kRecFp8);
        }
#pragma unroll 1
        for (int qq = 0; qq < 4; ++qq) {
          if (n_tile > 0) mbar_wait(&bars[kQuarterFree + qq], (n_tile - 1) & 1, abort_flag, p.d_error, kWaitLimitNs);
          // Store target: chunk 2qq + s8/4, row = token, 16-byte units
          // 2(s8&3) and 2(s8&3)+1; lanes 4-7 of each quarter-warp store the
          // odd unit first so that the 8 lanes of a phase hit 8 bank groups.
          uint8_t* chunk = sKV + (2 * qq + (s8 >> 2)) * 16384;
          const uint32_t u0 = 2 * (s8 & 3);
          const bool swap = (s8 & 4) != 0;
          auto store = [&](int r, const uint32_t (&o)[8]) {
            const uint32_t row = pw * 32 + r * 4 + j4;
            const uint4 a = make_uint4(o[0], o[1], o[2], o[3]);
            const uint4 b = make_uint4(o[4], o[5], o[6], o[7]);
            const uint32_t oa = swz<128>(row * 128 + u0 * 16);
            const uint32_t ob = swz<128>(row * 128 + (u0 + 1) * 16);
            *reinterpret_cast<uint4*>(chunk + (swap ? ob : oa)) = swap ? b : a;
            *reinterpret_cast<uint4*>(chunk + (swap ? oa : ob)) = swap ? a : b;
          };
          if (!ti.extra) {
            uint4 data[8];
            uint32_t sw[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              if (rec[r]) {
                data[r] = __ldg(reinterpret_cast<const uint4*>(rec[r] + qq * 128 + s8 * 16));
                sw[r] = __ldg(reinterpret_cast<const uint32_t*>(rec[r] + 512 + qq * 4));
              } else {
                data[r] = make_uint4(0, 0, 0, 0);
                sw[r] = 127u * 0x01010101u;
              }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              uint32_t o[8];
              dequant_fp8_16(data[r], (sw[r] >> (8 * (s8 >> 1))) & 0xFFu, o);
              store(r, o);
            }
          } else {
            uint2 data[8];
            uint32_t sb[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              if (rec[r]) {
                data[r] = __ldg(reinterpret_cast<const uint2*>(rec[r] + qq * 64 + s8 * 8));
                sb[r] = __ldg(rec[r] + 256 + qq * 8 + s8);
              } else {
                data[r] = make_uint2(0, 0);
                sb[r] = 0x38u;  // 1.0
              }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              uint32_t o[8];
              dequant_fp4_16(data[r].x, data[r].y, sb[r], o);
              store(r, o);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kQuarterFull + qq]);
        }
      }
      ++n_seg;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------
    // Tensor-core issuer (one thread).
    // ------------------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc_bf16(128, NH, false, false);
      constexpr uint32_t idesc_pv = make_idesc_bf16(128, NH, true, true);
      constexpr uint32_t p_row = 2 * NH;            // bytes per P^T row
      constexpr uint32_t p_sbo = 8 * p_row;         // 8-row group
      constexpr uint32_t p_swz = NH == 64 ? kSwizzle128 : (NH == 32 ? kSwizzle64 : kSwizzle32);
      const uint32_t kv_base = smem_u32(sKV), q_base = smem_u32(sQ), p_base = smem_u32(sP);
      const uint32_t tS = tmem, tO = tmem + NH;
      uint32_t n_tile = 0, n_seg = 0;
      bool issued = false;
      for (int64_t g = span.g_begin; g < span.g_end;) {
        const int qidx = static_cast<int>(g / p.T);
        const int64_t seg_end = min(span.g_end, static_cast<int64_t>(qidx + 1) * p.T);
        mbar_wait(&bars[kQFull], n_seg & 1, abort_flag, p.d_error, kWaitLimitNs);
        bool first = true;
        for (; g < seg_end; ++g, ++n_tile) {
          // S^T = K Q^T over the 8 dim chunks, as quarters arrive.
#pragma unroll 1
          for (int qq = 0; qq < 4; ++qq) {
            mbar_wait(&bars[kQuarterFull + qq], n_tile & 1, abort_flag, p.d_error, kWaitLimitNs);
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int c = 2 * qq + cc;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t a = make_smem_desc(kv_base + c * 16384 + k * 32, 16, 1024, kSwizzle128);
                const uint64_t b = make_smem_desc(q_base + c * (NH * 128) + k * 32, 16, 1024, kSwizzle128);
                mma_bf16_ss(tS, a, b, idesc_qk, (c | k) != 0);
              }
            }
          }
          issued = true;
          mma_commit(&bars[kSFull]);
          if (g + 1 == seg_end) mma_commit(&bars[kQFree]);
          // O^T += V^T P^T once the softmax has written P^T.
          mbar_wait(&bars[kPFull], n_tile & 1, abort_flag, p.d_error, kWaitLimitNs);
          tc_fence_after();
#pragma unroll 1
          for (int r = 0; r < 4; ++r) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t a = make_smem_desc(kv_base + 2 * r * 16384 + ks * 2048, 16384, 1024, kSwizzle128);
              const uint64_t b = make_smem_desc(p_base + ks * 2 * p_sbo, 16 * p_sbo, p_sbo, p_swz);
              mma_bf16_ss(tO + r * NH, a, b, idesc_pv, !(first && ks == 0));
            }
            mma_commit(&bars[kQuarterFree + r]);
          }
          if (g + 1 == seg_end) mma_commit(&bars[kOReady]);
          first = false;
        }
        ++n_seg;
      }
      if (issued) {
        // Normal runs have completed every product already (the softmax
        // waited for it); after a timeout this keeps TMEM alive until the
        // tensor core is done with it.
        mma_commit(&bars[kDrain]);
        mbar_wait(&bars[kDrain], 0, abort_flag, p.d_error, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------
    // Softmax and epilogue: thread i <-> TMEM lane i.
    // ------------------------------------------------------------------
    const int i = tid;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_base, tO = tmem + lane_base + NH;
    constexpr int V = NH >= 32 ? NH / 32 : 1;  // values a lane keeps after a reduce-scatter
    uint32_t n_tile = 0, n_seg = 0;
    if (i < NH) sm_m[i] = -INFINITY;
    for (int64_t g = span.g_begin; g < span.g_end;) {
      const int qidx = static_cast<int>(g / p.T);
      const int64_t seg_end = min(span.g_end, static_cast<int64_t>(qidx + 1) * p.T);
      const int64_t seg_begin = g;
      float lw[V];
#pragma unroll
      for (int k = 0; k < V; ++k) lw[k] = 0.f;
      for (; g < seg_end; ++g, ++n_tile) {
        const int t = static_cast<int>(g - static_cast<int64_t>(qidx) * p.T);
        const TileInfo ti = tile_info(p, qidx, t);
        const int slot = ti.slot0 + i;
        const int32_t id = slot < ti.nslots ? __ldg(ti.ids + slot) : -1;
        const bool valid = id >= 0 && static_cast<int64_t>(id) < ti.pool;

        mbar_wait(&bars[kSFull], n_tile & 1, abort_flag, p.d_error, kWaitLimitNs);
        tc_fence_after();
        // Column max over the 128 tokens of the tile (reduce-scatter in place).
        {
          float v[NH];
#pragma unroll
          for (int c = 0; c < NH / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(tS + c * 16, r);
#pragma unroll
            for (int k = 0; k < 16; ++k) v[c * 16 + k] = valid ? __uint_as_float(r[k]) * p.scale_log2 : -INFINITY;
          }
          ReduceScatter<NH, 16>::run(v, lane, MaxOp());
#pragma unroll
          for (int k = 0; k < V; ++k) red[warp * NH + rs_head<NH>(lane, k)] = v[k];
        }
        named_bar_sync(1, kSoftmaxThreads);
        int need = 0;
        if (i < NH) {
          const float mt = fmaxf(fmaxf(red[i], red[NH + i]), fmaxf(red[2 * NH + i], red[3 * NH + i]));
          const float m_old = sm_m[i];
          float alpha = 1.f;
          if (mt > m_old + kLazyRescale || (m_old == -INFINITY && mt > -INFINITY)) {
            alpha = m_old == -INFINITY ? 0.f : ex2_approx(m_old - mt);
            need = m_old != -INFINITY;
            sm_m[i] = mt;
          }
          sm_alpha[i] = alpha;
        }
        int any_rescale;
        asm volatile(
            "{\n\t.reg .pred pi, po;\n\t"
            "setp.ne.s32 pi, %1, 0;\n\t"
            "bar.red.or.pred po, 2, %2, pi;\n\t"
            "selp.s32 %0, 1, 0, po;\n\t}"
            : "=r"(any_rescale)
            : "r"(need), "r"(kSoftmaxThreads)
            : "memory");
        // P = 2^(x - m) (S re-read from TMEM), stored as row i of P^T
        // (MN-major, swizzled), then its column sums.
        {
          float v[NH];
#pragma unroll
          for (int c = 0; c < NH / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(tS + c * 16, r);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float m = sm_m[c * 16 + k];
              const float xv = __uint_as_float(r[k]) * p.scale_log2;
              v[c * 16 + k] = (!valid || m == -INFINITY) ? 0.f : ex2_approx(xv - m);
            }
          }
#pragma unroll
          for (int u = 0; u < NH / 8; ++u) {
            uint4 w;
            w.x = pack_bf16x2(v[8 * u + 0], v[8 * u + 1]);
            w.y = pack_bf16x2(v[8 * u + 2], v[8 * u + 3]);
            w.z = pack_bf16x2(v[8 * u + 4], v[8 * u + 5]);
            w.w = pack_bf16x2(v[8 * u + 6], v[8 * u + 7]);
            *reinterpret_cast<uint4*>(sP + swz<2 * NH>(i * (2 * NH) + u * 16)) = w;
          }
          ReduceScatter<NH, 16>::run(v, lane, AddOp());
#pragma unroll
          for (int k = 0; k < V; ++k) lw[k] = lw[k] * sm_alpha[rs_head<NH>(lane, k)] + v[k];
        }
        if (any_rescale) {
          // O^T[d, h] *= alpha[h]; the previous products are complete
          // (the tensor core finished them before this tile's S^T).
#pragma unroll 1
          for (int r = 0; r < 4; ++r) {
#pragma unroll
            for (int c = 0; c < NH / 16; ++c) {
              uint32_t o[16];
              tmem_ld16(tO + r * NH + c * 16, o);
              #pragma unroll
              for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * sm_alpha[c * 16 + k]);
              tmem_st16(tO + r * NH + c * 16, o);
            }
          }
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[kPFull]);
      }
      // Epilogue of this query token (or of this split of it).
      mbar_wait(&bars[kOReady], n_seg & 1, abort_flag, p.d_error, kWaitLimitNs);
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < V; ++k) red[warp * NH + rs_head<NH>(lane, k)] = lw[k];
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
      ++n_seg;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace

template <int NH>
cudaError_t launch_decode(const DecodeParams& p, int grid, cudaStream_t stream) {
  constexpr int smem = Smem<NH>::kAlloc;
  static bool configured = false;  // benign race: the attribute call is idempotent
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(sparse_decode_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  sparse_decode_kernel<NH><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template cudaError_t launch_decode<16>(const DecodeParams&, int, cudaStream_t);
template cudaError_t launch_decode<32>(const DecodeParams&, int, cudaStream_t);
template cudaError_t launch_decode<64>(const DecodeParams&, int, cudaStream_t);

int decode_smem_bytes(int nh) {
  return nh == 64 ? Smem<64>::kAlloc : (nh == 32 ? Smem<32>::kAlloc : Smem<16>::kAlloc);
}

}  // namespace mla
