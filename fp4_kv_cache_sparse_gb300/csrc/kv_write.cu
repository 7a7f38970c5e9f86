// kv_write.cu -- the KV-cache writer: quantize new tokens' 512-dim latents
// (bf16) into records of the paged pool and store each at its slot
// (page * 64 + offset).  The record formats are those of
// "flops/flashmla-decode-fp8-fp4-kv", "Arithmetic intensity": 528 bytes of
// e4m3 data plus one e8m0 scale per 32 values, or 288 bytes of e2m1 data
// (even index in the low nibble) plus one e4m3 scale per 16 values.  The
// block scale rule (the pages give only "amax"-style scaling): FP8 takes the
// least power of two 2^e with amax * 2^-e <= 448 (byte 127 + e, 127 for an
// all-zero block, e clamped to [-127, 127]); FP4 takes amax / 6 rounded to
// E4M3FN.  Every element rounds to nearest, ties to even, saturating.
//
// One warp per token.  FP8: lane l holds dims 16l .. 16l+15, half of a
// 32-value block (the block maximum is one shuffle); FP4: lane l holds the
// 16-value block l.  Conversions are the hardware's round-to-nearest-even
// cvt.rn.satfinite to e4m3x2 / e2m1x2; the scalings before them are exact
// (a power of two, or an IEEE division whose rounding cannot move a bf16
// quotient across a rounding boundary of the 2- or 4-bit target).
#include <cstdint>
#include <cuda_fp16.h>

#include "../../include/mla.h"
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kWarps = 8;
constexpr int kRecFp8Bytes = 528;
constexpr int kRecFp4Bytes = 288;

// Eight floats -> eight e2m1 nibbles (x[0] in the low nibble of byte 0).
__device__ __forceinline__ uint32_t e2m1x8(const float (&x)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return r;
}

// E4M3FN byte -> float, exactly (through f16, which holds every e4m3 value).
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(byte)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// 16 bf16 values of this lane (dims 16 lane .. 16 lane + 15) as floats.
__device__ __forceinline__ void load16(const uint16_t* src, float (&x)[16]) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
  const uint4 a = __ldg(p), b = __ldg(p + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(kWarps * 32) kv_write_fp8_kernel(const uint16_t* __restrict__ lat,
                                                                   const int32_t* __restrict__ slots, int64_t n,
                                                                   uint8_t* __restrict__ pool, int64_t pool_tokens,
                                                                   int32_t* d_error) {
  const int lane = threadIdx.x & 31;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); t < n;
       t += static_cast<int64_t>(gridDim.x) * kWarps) {
    const int32_t slot = __ldg(slots + t);
    if (slot < 0 || slot >= pool_tokens) {
      if (slot != -1 && lane == 0 && d_error) atomicOr(d_error, MLA_DEVERR_BAD_INDEX);
      continue;
    }
    float x[16];
    load16(lat + t * MLA_HEAD_DIM + 16 * lane, x);
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));  // the 32-value block of lanes 2b, 2b+1
    const int e = fp8_block_exponent(amax);
    uint32_t q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      q[k] = e4m3x2(ldexpf(x[4 * k], -e), ldexpf(x[4 * k + 1], -e)) |
             (e4m3x2(ldexpf(x[4 * k + 2], -e), ldexpf(x[4 * k + 3], -e)) << 16);
    uint8_t* rec = pool + static_cast<int64_t>(slot) * kRecFp8Bytes;
    *reinterpret_cast<uint4*>(rec + 16 * lane) = make_uint4(q[0], q[1], q[2], q[3]);
    // Scale bytes of blocks 4m .. 4m+3 gathered by lane m (m < 4), one 4-byte store each.
    const uint32_t sb = static_cast<uint32_t>(127 + e);
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) word |= __shfl_sync(0xFFFFFFFFu, sb, (8 * lane + 2 * k) & 31) << (8 * k);
    if (lane < 4) *reinterpret_cast<uint32_t*>(rec + MLA_HEAD_DIM + 4 * lane) = word;
  }
}

__global__ void __launch_bounds__(kWarps * 32) kv_write_fp4_kernel(const uint16_t* __restrict__ lat,
                                                                   const int32_t* __restrict__ slots, int64_t n,
                                                                   uint8_t* __restrict__ pool, int64_t pool_tokens,
                                                                   int32_t* d_error) {
  const int lane = threadIdx.x & 31;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); t < n;
       t += static_cast<int64_t>(gridDim.x) * kWarps) {
    const int32_t slot = __ldg(slots + t);
    if (slot < 0 || slot >= pool_tokens) {
      if (slot != -1 && lane == 0 && d_error) atomicOr(d_error, MLA_DEVERR_BAD_INDEX);
      continue;
    }
    float x[16];
    load16(lat + t * MLA_HEAD_DIM + 16 * lane, x);
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
    const uint32_t sc = e4m3x2(__fdiv_rn(amax, 6.f), 0.f) & 0xFFu;
    const float s = e4m3_to_float(sc);
    uint32_t q[2] = {0u, 0u};
    if (s != 0.f) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float y[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = __fdiv_rn(x[8 * h + k], s);
        q[h] = e2m1x8(y);
      }
    }
    uint8_t* rec = pool + static_cast<int64_t>(slot) * kRecFp4Bytes;
    *reinterpret_cast<uint2*>(rec + 8 * lane) = make_uint2(q[0], q[1]);
    // Scale bytes 4m .. 4m+3 gathered by lane m (m < 8).
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) word |= __shfl_sync(0xFFFFFFFFu, sc, (4 * lane + k) & 31) << (8 * k);
    if (lane < 8) *reinterpret_cast<uint32_t*>(rec + 256 + 4 * lane) = word;
  }
}

}  // namespace

cudaError_t launch_kv_write(int kv_format, const uint16_t* latents, const int32_t* slots, int64_t n, uint8_t* pool,
                            int64_t pool_tokens, int32_t* d_error, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (blocks > cap) blocks = cap;
  if (kv_format == MLA_KV_FP8_528)
    kv_write_fp8_kernel<<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(latents, slots, n, pool,
                                                                                    pool_tokens, d_error);
  else
    kv_write_fp4_kernel<<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(latents, slots, n, pool,
                                                                                    pool_tokens, d_error);
  return cudaGetLastError();
}

}  // namespace mla
