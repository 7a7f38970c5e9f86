// combine.cu -- merge of split-KV partials by their log-sum-exp
// ("flops/flashmla-decode-fp8-fp4-kv", "Workarounds": split decoding with
// num_splits).  One warp per (query token, head).  The lanes split the
// splits: lane j reads the LSEs of splits j, j+32, ..., the maximum and the
// sum of exp(lse_i - max) are warp-shuffle reductions, and lane j keeps the
// weight of its splits.  The weighted sum then walks the splits in pairs,
// each lane accumulating 16 of the 512 dims from float4 loads that are all
// issued before any is used.  Blocks of four warps at no more than 73
// registers a thread (seven blocks a SM), so that the rows of a 64-query,
// 64-head batch are all resident at once.  In the grid over the decode's
// parts (a block = four heads of one split query token, which then has at
// most two splits) the block's partial rows come by bulk copies into shared
// memory, issued before the LSE loads.
#include <cstdint>
#include <cuda_bf16.h>

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kWarps = 4;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// The merged output of one (query token, head) row: lane l ends with dims
// 128 k + 4 l .. 128 k + 4 l + 3 in acc[4 k .. 4 k + 3]; returns the row's
// log-sum-exp (natural log; -inf when every split is empty, acc all zero).
__device__ __forceinline__ float merge_row(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                                           int s0, int n, int h, int h_q, int lane, float (&acc)[16]) {
  const float* lrow = lse_part + static_cast<int64_t>(s0) * h_q + h;
  // Max and sum over the splits, lanes striding over them.
  float mx = -INFINITY;
  for (int i = lane; i < n; i += 32) mx = fmaxf(mx, lrow[static_cast<int64_t>(i) * h_q]);
  const float M = warp_max(mx);
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  if (M == -INFINITY) return -INFINITY;
  float z = 0.f;
  for (int i = lane; i < n; i += 32) {
    const float li = lrow[static_cast<int64_t>(i) * h_q];
    z += li == -INFINITY ? 0.f : expf(li - M);
  }
  const float L = M + logf(warp_sum(z));
  const float* orow = o_part + (static_cast<int64_t>(s0) * h_q + h) * 512;
  const int64_t ostride = static_cast<int64_t>(h_q) * 512;
  for (int c = 0; c < n; c += 32) {
    // Weight of split c + lane, held by that lane; -inf partials weigh 0.
    float wl = 0.f;
    if (c + lane < n) {
      const float li = lrow[static_cast<int64_t>(c + lane) * h_q];
      wl = li == -INFINITY ? 0.f : expf(li - L);
    }
    const int m = min(32, n - c);
    for (int j = 0; j < m; j += 2) {
      float4 v[2][4];
      float w[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        w[u] = __shfl_sync(kFull, wl, (j + u) & 31);
        const bool use = j + u < m && w[u] != 0.f;
        const float4* src = reinterpret_cast<const float4*>(orow + (c + j + u) * ostride);
#pragma unroll
        for (int k = 0; k < 4; ++k) v[u][k] = use ? src[k * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        if (!use) w[u] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[4 * k + 0] += w[u] * v[u][k].x;
          acc[4 * k + 1] += w[u] * v[u][k].y;
          acc[4 * k + 2] += w[u] * v[u][k].z;
          acc[4 * k + 3] += w[u] * v[u][k].w;
        }
      }
    }
  }
  return L;
}

// The query token and head of this warp.  kByPart: blockIdx.x is a part of
// the decode's schedule and blockIdx.y a group of kWarps heads; the only
// query token of a part that can have several splits is the one holding the
// part's last tile, and it is merged by the part in which it starts (so
// once); -1 when the part has nothing to merge.  Otherwise one warp per
// (query token, head) row, every token visited.
template <bool kByPart>
__device__ __forceinline__ int64_t merge_row_of(const int32_t* __restrict__ sched, int T, int h_q, int& h) {
  const int warp = threadIdx.x >> 5;
  if constexpr (!kByPart) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    h = static_cast<int>(row % h_q);
    return row / h_q;
  }
  const int32_t* e = sched + static_cast<int64_t>(blockIdx.x) * MLA_SCHED_INTS;
  const int64_t g0 = e[0], g1 = e[1];
  h = static_cast<int>(blockIdx.y) * kWarps + warp;
  if (g1 <= g0 || T <= 0) return -1;
  const int64_t q = (g1 - 1) / T;
  return q * T >= g0 ? q : -1;
}

// The by-part grid's merge of one split query token for the block's four
// heads: their partial rows of each split (4 x 2 KB, contiguous) arrive by
// one bulk copy per split into shared memory, issued before the LSE loads so
// that the two overlap.  Returns false (nothing done) when there are more
// splits than the staging holds.
constexpr int kStageSplits = 2;
__device__ __forceinline__ bool merge_rows_staged(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                                                  int s0, int n, int h0, int h_q, float (&acc)[16], float& L) {
  __shared__ alignas(128) float stage[kStageSplits][kWarps * 512];
  __shared__ alignas(8) uint64_t bar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (n > kStageSplits) return false;
  const int nh = min(kWarps, h_q - h0);
  const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(n * nh * 2048) : "memory");
    for (int i = 0; i < n; ++i)
      asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                       static_cast<uint32_t>(__cvta_generic_to_shared(&stage[i][0]))),
                   "l"(o_part + (static_cast<int64_t>(s0 + i) * h_q + h0) * 512), "r"(nh * 2048), "r"(b)
                   : "memory");
  }
  __syncthreads();
  const int h = h0 + warp;
  const float* lrow = lse_part + static_cast<int64_t>(s0) * h_q + h;
  const float li = lane < n ? lrow[static_cast<int64_t>(lane) * h_q] : -INFINITY;
  const float M = warp_max(li);
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float wl = 0.f;
  if (M != -INFINITY) {
    const float z = li == -INFINITY ? 0.f : expf(li - M);
    L = M + logf(warp_sum(z));
    wl = li == -INFINITY ? 0.f : expf(li - L);
  } else {
    L = -INFINITY;
  }
  // The copies land (bounded wait: 2 s of global time, then the block goes
  // on; they cannot fail short of a fault).
  {
    uint32_t ok = 0;
    uint64_t t0 = 0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(b)
          : "memory");
      if (ok) break;
      uint64_t t1;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
      if (t1 - t0 > 2000000000ull) break;
    }
  }
  if (M == -INFINITY || warp >= nh) return true;
  for (int i = 0; i < n; ++i) {
    const float w = __shfl_sync(kFull, wl, i);
    if (w == 0.f) continue;
    const float4* src = reinterpret_cast<const float4*>(&stage[i][warp * 512]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 v = src[k * 32 + lane];
      acc[4 * k + 0] += w * v.x;
      acc[4 * k + 1] += w * v.y;
      acc[4 * k + 2] += w * v.z;
      acc[4 * k + 3] += w * v.w;
    }
  }
  return true;
}

template <bool kByPart>
__global__ void __launch_bounds__(kWarps * 32, 7) combine_kernel(const int32_t* __restrict__ num_splits,
                                                             const float* __restrict__ o_part,
                                                             const float* __restrict__ lse_part,
                                                             uint16_t* __restrict__ out, float* __restrict__ lse,
                                                             int nq, int h_q, int skip_single,
                                                             const int32_t* __restrict__ sched, int T) {
  // Launched as a programmatic dependent of the decode kernel: wait until
  // that grid has completed and its partials are visible (returns at once
  // for an ordinary launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  int h;
  const int64_t q = merge_row_of<kByPart>(sched, T, h_q, h);
  if (q < 0 || q >= nq || h >= h_q) return;  // whole warps leave together
  const int qidx = static_cast<int>(q);
  const int64_t row = q * h_q + h;
  const int s0 = num_splits[qidx];
  const int n = num_splits[qidx + 1] - s0;
  if (skip_single && n == 1) return;
  float acc[16];
  float L;
  bool staged = false;
  if constexpr (kByPart)
    staged = merge_rows_staged(o_part, lse_part, s0, n, static_cast<int>(blockIdx.y) * kWarps, h_q, acc, L);
  if (!staged) L = merge_row(o_part, lse_part, s0, n, h, h_q, lane, acc);
  uint2* dst = reinterpret_cast<uint2*>(out + row * 512);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc[4 * k + 0], acc[4 * k + 1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[4 * k + 2], acc[4 * k + 3]);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&a);
    w.y = *reinterpret_cast<const uint32_t*>(&b);
    dst[k * 32 + lane] = w;
  }
  if (lane == 0) lse[row] = L;
}

// The fused output epilogue ("deepseek-ai/FlashMLA", "What it is": the
// conjugate RoPE on the output side and the cast to FP8).  Every query
// token's splits (one or more; with skip_single only tokens of several
// splits, the 128-head decode kernel having written the others with the
// same arithmetic) are merged as above; then dims 448..511 (the
// rotary part: 32 interleaved pairs, held by lanes 16..31 in acc[12..15])
// turn by -phi_j, phi_j = pos * theta^(-2j/64) (rope_cos_sin, rope_conj_apply); then each
// 32-dim block (eight lanes) is cast to E4M3FN under its e8m0 scale, giving
// a 528-byte record per row in the cache's own format.
template <bool kByPart>
__global__ void __launch_bounds__(kWarps * 32, 4) rope_fp8_kernel(const int32_t* __restrict__ num_splits,
                                                              const float* __restrict__ o_part,
                                                              const float* __restrict__ lse_part,
                                                              const int32_t* __restrict__ positions,
                                                              const RopeFreqs freqs, uint8_t* __restrict__ out,
                                                              float* __restrict__ lse, int nq, int h_q,
                                                              int skip_single, const int32_t* __restrict__ sched,
                                                              int T) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  int h;
  const int64_t q = merge_row_of<kByPart>(sched, T, h_q, h);
  if (q < 0 || q >= nq || h >= h_q) return;  // whole warps leave together
  const int qidx = static_cast<int>(q);
  const int64_t row = q * h_q + h;
  const int s0 = num_splits[qidx];
  const int n = num_splits[qidx + 1] - s0;
  if (skip_single && n == 1) return;  // written by the decode kernel itself
  float acc[16];
  float L;
  bool staged = false;
  if constexpr (kByPart)
    staged = merge_rows_staged(o_part, lse_part, s0, n, static_cast<int>(blockIdx.y) * kWarps, h_q, acc, L);
  if (!staged) L = merge_row(o_part, lse_part, s0, n, h, h_q, lane, acc);
  if (lane >= 16) {
    const double pos = static_cast<double>(positions[qidx]);
#pragma unroll
    for (int u = 0; u < 2; ++u) {  // pair (448 + 2j, 449 + 2j), j = 2 (lane - 16) + u
      float cs, sn;
      rope_cos_sin(pos, freqs.f[2 * (lane - 16) + u], cs, sn);
      rope_conj_apply(acc[12 + 2 * u], acc[13 + 2 * u], cs, sn);
    }
  }
  uint8_t* rec = out + row * 528;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    // Block 4 k + lane / 8: its eight lanes agree on the maximum.
    float amax = fmaxf(fmaxf(fabsf(acc[4 * k]), fabsf(acc[4 * k + 1])), fmaxf(fabsf(acc[4 * k + 2]), fabsf(acc[4 * k + 3])));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
    const int e = fp8_block_exponent(amax);
    const uint32_t word = e4m3x2(ldexpf(acc[4 * k], -e), ldexpf(acc[4 * k + 1], -e)) |
                          (e4m3x2(ldexpf(acc[4 * k + 2], -e), ldexpf(acc[4 * k + 3], -e)) << 16);
    *reinterpret_cast<uint32_t*>(rec + 128 * k + 4 * lane) = word;
    if ((lane & 7) == 0) rec[512 + 4 * k + (lane >> 3)] = static_cast<uint8_t>(127 + e);
  }
  if (lane == 0) lse[row] = L;
}

}  // namespace

// One warp per row (sched == null), or parts x head groups (only the rows of
// split query tokens; the caller guarantees that every other row was written
// by the decode kernel itself).
static void merge_grid(int64_t rows, const int32_t* sched, int num_parts, int h_q, dim3& grid) {
  if (sched != nullptr)
    grid = dim3(static_cast<unsigned>(num_parts), static_cast<unsigned>((h_q + kWarps - 1) / kWarps));
  else
    grid = dim3(static_cast<unsigned>((rows + kWarps - 1) / kWarps));
}

cudaError_t launch_combine(const int32_t* d_num_splits, const float* o_part, const float* lse_part, uint16_t* out,
                           float* lse, int nq, int h_q, bool skip_single, const int32_t* sched, int num_parts, int T,
                           cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(nq) * h_q;
  if (rows == 0 || (sched != nullptr && num_parts <= 0)) return cudaSuccess;
  // Programmatic stream serialization: the merge's blocks may be scheduled
  // while the preceding kernel drains; each waits for it (griddepcontrol)
  // before reading anything.
  cudaLaunchConfig_t cfg{};
  merge_grid(rows, sched, num_parts, h_q, cfg.gridDim);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (sched != nullptr)
    return cudaLaunchKernelEx(&cfg, combine_kernel<true>, d_num_splits, o_part, lse_part, out, lse, nq, h_q,
                              skip_single ? 1 : 0, sched, T);
  return cudaLaunchKernelEx(&cfg, combine_kernel<false>, d_num_splits, o_part, lse_part, out, lse, nq, h_q,
                            skip_single ? 1 : 0, sched, T);
}

cudaError_t launch_rope_fp8(const int32_t* d_num_splits, const float* o_part, const float* lse_part,
                            const int32_t* positions, const RopeFreqs& freqs, uint8_t* out, float* lse, int nq,
                            int h_q, bool skip_single, const int32_t* sched, int num_parts, int T,
                            cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(nq) * h_q;
  if (rows == 0 || (sched != nullptr && num_parts <= 0)) return cudaSuccess;
  cudaLaunchConfig_t cfg{};
  merge_grid(rows, sched, num_parts, h_q, cfg.gridDim);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (sched != nullptr)
    return cudaLaunchKernelEx(&cfg, rope_fp8_kernel<true>, d_num_splits, o_part, lse_part, positions, freqs, out,
                              lse, nq, h_q, skip_single ? 1 : 0, sched, T);
  return cudaLaunchKernelEx(&cfg, rope_fp8_kernel<false>, d_num_splits, o_part, lse_part, positions, freqs, out, lse,
                            nq, h_q, skip_single ? 1 : 0, sched, T);
}

}  // namespace mla
