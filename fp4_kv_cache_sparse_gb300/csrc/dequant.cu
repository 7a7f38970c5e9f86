// dequant.cu -- whole-record dequantization with the decode kernel's own
// device routines (dequant_fp8_16 / dequant_fp4_16), one thread per 16
// dims.  ("flops/flashmla-decode-fp8-fp4-kv", "Arithmetic intensity".)
#include <cstdint>

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

namespace {

__global__ void __launch_bounds__(256) dequant_kernel(int kv_format, const uint8_t* __restrict__ records, int64_t n,
                                                      uint16_t* __restrict__ out) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // Whole warps stay active (the decode kernel picks its FP8 routine with a
  // warp vote; this kernel makes the same choice the same way).
  const bool live = t < n * 32;
  const int64_t tt = live ? t : 0;
  const int64_t r = tt >> 5;
  const int seg = static_cast<int>(tt & 31);  // dims 16*seg .. 16*seg+15
  uint32_t v[8];
  if (kv_format == MLA_KV_FP8_528) {
    const uint8_t* rec = records + r * kRecFp8;
    const uint4 data = __ldg(reinterpret_cast<const uint4*>(rec + seg * 16));
    const uint32_t sbyte = rec[512 + seg / 2];
    if (__any_sync(0xFFFFFFFFu, sbyte > 142u))
      dequant_fp8_16(data, sbyte, v);
    else
      dequant_fp8_16_small_scale(data, sbyte, v);
  } else {
    const uint8_t* rec = records + r * kRecFp4;
    const uint2 data = __ldg(reinterpret_cast<const uint2*>(rec + seg * 8));
    dequant_fp4_16(data.x, data.y, rec[256 + seg], v);
  }
  if (!live) return;
  uint4* dst = reinterpret_cast<uint4*>(out + r * kD + seg * 16);
  dst[0] = make_uint4(v[0], v[1], v[2], v[3]);
  dst[1] = make_uint4(v[4], v[5], v[6], v[7]);
}

}  // namespace

cudaError_t launch_dequant(int kv_format, const uint8_t* records, int64_t n, uint16_t* out, cudaStream_t stream) {
  const int64_t threads = n * 32;
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = (threads + 255) / 256;
  dequant_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(kv_format, records, n, out);
  return cudaGetLastError();
}

}  // namespace mla
