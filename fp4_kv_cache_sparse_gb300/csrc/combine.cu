// combine.cu -- merge of split-KV partials by their log-sum-exp
// ("flops/flashmla-decode-fp8-fp4-kv", "Workarounds": split decoding with
// num_splits).  One warp per (query token, head): the split weights come
// from a max and a sum over the splits' LSEs, then each lane accumulates 16
// of the 512 dims from float4 loads.
#include <cstdint>
#include <cuda_bf16.h>

#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) combine_kernel(const int32_t* __restrict__ num_splits,
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
  if (row >= static_cast<int64_t>(nq) * h_q) return;
  const int qidx = static_cast<int>(row / h_q);
  const int h = static_cast<int>(row % h_q);
  const int s0 = num_splits[qidx];
  const int n = num_splits[qidx + 1] - s0;
  if (skip_single && n == 1) return;

  float M = -INFINITY;
  for (int i = 0; i < n; ++i) M = fmaxf(M, lse_part[static_cast<int64_t>(s0 + i) * h_q + h]);
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float L = -INFINITY;
  if (M != -INFINITY) {
    float Z = 0.f;
    for (int i = 0; i < n; ++i) Z += expf(lse_part[static_cast<int64_t>(s0 + i) * h_q + h] - M);
    L = M + logf(Z);
    for (int i = 0; i < n; ++i) {
      const float li = lse_part[static_cast<int64_t>(s0 + i) * h_q + h];
      if (li == -INFINITY) continue;
      const float w = expf(li - L);
      const float4* src = reinterpret_cast<const float4*>(o_part + (static_cast<int64_t>(s0 + i) * h_q + h) * 512);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 v = src[k * 32 + lane];
        acc[4 * k + 0] += w * v.x;
        acc[4 * k + 1] += w * v.y;
        acc[4 * k + 2] += w * v.z;
        acc[4 * k + 3] += w * v.w;
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
