// combine.cu -- merge of split-KV partials by their log-sum-exp
// ("flops/flashmla-decode-fp8-fp4-kv", "Workarounds": split decoding with
// num_splits).  One warp per (query token, head).  The lanes split the
// splits: lane j reads the LSEs of splits j, j+32, ..., the maximum and the
// sum of exp(lse_i - max) are warp-shuffle reductions, and lane j keeps the
// weight of its splits.  The weighted sum then walks the splits in pairs,
// each lane accumulating 16 of the 512 dims from float4 loads that are all
// issued before any is used.  Blocks of four warps at no more than 73
// registers a thread (seven blocks a SM), so that the rows of a 64-query,
// 64-head batch are all resident at once.
#include <cstdint>
#include <cuda_bf16.h>

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

__global__ void __launch_bounds__(kWarps * 32, 7) combine_kernel(const int32_t* __restrict__ num_splits,
                                                             const float* __restrict__ o_part,
                                                             const float* __restrict__ lse_part,
                                                             uint16_t* __restrict__ out, float* __restrict__ lse,
                                                             int nq, int h_q, int skip_single) {
  // Launched as a programmatic dependent of the decode kernel: wait until
  // that grid has completed and its partials are visible (returns at once
  // for an ordinary launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= static_cast<int64_t>(nq) * h_q) return;  // whole warps leave together
  const int qidx = static_cast<int>(row / h_q);
  const int h = static_cast<int>(row % h_q);
  const int s0 = num_splits[qidx];
  const int n = num_splits[qidx + 1] - s0;
  if (skip_single && n == 1) return;
  const float* lrow = lse_part + static_cast<int64_t>(s0) * h_q + h;

  // Max and sum over the splits, lanes striding over them.
  float mx = -INFINITY;
  for (int i = lane; i < n; i += 32) mx = fmaxf(mx, lrow[static_cast<int64_t>(i) * h_q]);
  const float M = warp_max(mx);
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float L = -INFINITY;
  if (M != -INFINITY) {
    float z = 0.f;
    for (int i = lane; i < n; i += 32) {
      const float li = lrow[static_cast<int64_t>(i) * h_q];
      z += li == -INFINITY ? 0.f : expf(li - M);
    }
    L = M + logf(warp_sum(z));
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
  }
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

}  // namespace

cudaError_t launch_combine(const int32_t* d_num_splits, const float* o_part, const float* lse_part, uint16_t* out,
                           float* lse, int nq, int h_q, bool skip_single, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(nq) * h_q;
  const int64_t blocks = (rows + kWarps - 1) / kWarps;
  if (blocks == 0) return cudaSuccess;
  // Programmatic stream serialization: the merge's blocks may be scheduled
  // while the preceding kernel drains; each waits for it (griddepcontrol)
  // before reading anything.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, d_num_splits, o_part, lse_part, out, lse, nq, h_q,
                            skip_single ? 1 : 0);
}

}  // namespace mla
