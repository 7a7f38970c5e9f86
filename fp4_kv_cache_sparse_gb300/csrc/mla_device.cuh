// mla_device.cuh -- device-side building blocks for the sm_103a decode path:
// inline-PTX wrappers for mbarriers, tcgen05 (TMEM allocation, MMA, loads),
// shared-memory matrix descriptors, the 128-byte swizzle, and the exact
// in-register dequantization of the FP8 (528 B) and FP4 (288 B) token records
// ("flops/flashmla-decode-fp8-fp4-kv", section "Arithmetic intensity").
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kD = 512;          // latent width
constexpr int kPage = 64;        // tokens per page
constexpr int kRecFp8 = 528;     // 512 B e4m3 + 16 B e8m0
constexpr int kRecFp4 = 288;     // 256 B e2m1 + 32 B e4m3
constexpr int kTile = 128;       // index slots per tile (= MMA M)

// ---------------------------------------------------------------------------
// Small PTX helpers.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Gives up after `limit_ns` of global
// time (or at once when another thread of the CTA has already given up),
// records MLA_DEVERR_TIMEOUT and returns false; the caller carries on so that
// every thread still reaches the CTA-wide barriers and the kernel ends.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* d_error, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        if (d_error) atomicOr(d_error, MLA_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Make this thread's generic-proxy shared-memory writes visible to the
// async proxy (the tensor core reads its operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor core.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on an mbarrier once every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 16 columns of 32-bit TMEM words: thread i of the warp gets lane
// (warp quadrant base + i), columns col..col+15.  The load and its
// completion wait are one asm statement so that no use of the registers can
// be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"):
//   [0,14)  start address >> 4        [16,30) leading byte offset >> 4
//   [32,46) stride byte offset >> 4    [46,49) fixed 0b001
//   [49,52) base offset (0: atoms aligned)   [61,64) swizzle mode
enum : uint32_t { kSwizzleNone = 0, kSwizzle128 = 2, kSwizzle64 = 4, kSwizzle32 = 6 };

__device__ __forceinline__ uint64_t make_smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                                   uint32_t swizzle) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFF) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle & 0x7) << 61;
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A/B and fp32 D.
//   [4,6) D format (1 = f32)   [7,10) A format (1 = bf16)   [10,13) B format
//   [15] A major (1 = MN)      [16] B major (1 = MN)
//   [17,23) N >> 3             [24,29) M >> 4
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Swizzled byte offset inside a 1024-byte-aligned region whose rows are
// `row_bytes` wide (128, 64 or 32): the 16-byte unit index (bits 4..6) is
// XOR-ed with the row bits 7..9 masked to the swizzle width.
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  constexpr uint32_t mask = ROW_BYTES == 128 ? 7u : (ROW_BYTES == 64 ? 3u : 1u);
  return off ^ (((off >> 7) & mask) << 4);
}

// ---------------------------------------------------------------------------
// Exact dequantization, 16 values at a time ("Arithmetic intensity").
// ---------------------------------------------------------------------------

// bf16x2 product, rounded once to nearest even.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two e4m3 bytes (low 16 bits of w) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w16) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(r) : "r"(w16));
  return r;
}

// Two e2m1 values (low byte of w) -> f16x2, exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t w8) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(w8));
  return r;
}

// f16x2 whose values need at most 8 significant bits and lie in the f16
// normal range (or are zero) -> bf16x2 bit patterns of value * 2^-112.
// Shifting right by 3 re-reads the 5-bit f16 exponent as a bf16 exponent
// with a bias 112 larger and keeps the top 7 mantissa bits; the low mantissa
// bits of both halves are zero for such values, so each sign bit lands 3
// places low with zeros above it, and adding 7 times it carries it home.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_scaled(uint32_t h) {
  const uint32_t u = h >> 3;
  return u + (u & 0x10001000u) * 7u;
}

__device__ __forceinline__ uint32_t bf16x2_splat_pow2(int e) {  // 2^e as bf16x2, e in [-126, 127]
  const uint32_t b = static_cast<uint32_t>(e + 127) << 7;
  return b | (b << 16);
}

// Four e4m3 bytes -> two bf16x2 patterns of value * 2^-112 (dims 0,1 / 2,3).
__device__ __forceinline__ void e4m3x4_to_bf16x2x2_scaled(uint32_t w, uint32_t& lo, uint32_t& hi) {
  uint32_t a, b;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(a), "=r"(b)
      : "r"(w));
  lo = f16x2_to_bf16x2_scaled(a);
  hi = f16x2_to_bf16x2_scaled(b);
}

// 16 consecutive dims of an FP8 record: data = 16 e4m3 bytes, sbyte = the
// e8m0 scale byte of their 32-dim block.  value = e4m3 * 2^(sbyte-127),
// rounded once to bf16 (exact whenever the product is a normal bf16).
// out[i] packs dims (2i, 2i+1) as bf16x2 (low half = even dim).
// Valid for every scale byte; two multiplies when sbyte > 142.
__device__ __forceinline__ void dequant_fp8_16(const uint4& data, uint32_t sbyte, uint32_t (&out)[8]) {
  // pattern = value * 2^-112; then * 2^(112 + sbyte - 127).
  const int e = static_cast<int>(sbyte) - 15;
  const bool two_step = e > 127;
  const uint32_t c1 = bf16x2_splat_pow2(two_step ? 127 : e);
  const uint32_t c2 = bf16x2_splat_pow2(two_step ? e - 127 : 0);
  const uint32_t w[4] = {data.x, data.y, data.z, data.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t lo, hi;
    e4m3x4_to_bf16x2x2_scaled(w[k], lo, hi);
    lo = bf16x2_mul(lo, c1);
    hi = bf16x2_mul(hi, c1);
    if (two_step) {
      lo = bf16x2_mul(lo, c2);
      hi = bf16x2_mul(hi, c2);
    }
    out[2 * k] = lo;
    out[2 * k + 1] = hi;
  }
}

// The same for scale bytes <= 142 (scales up to 2^15): one multiply.  Gives
// results identical to dequant_fp8_16 on that range.
__device__ __forceinline__ void dequant_fp8_16_small_scale(const uint4& data, uint32_t sbyte, uint32_t (&out)[8]) {
  const uint32_t c = (sbyte + 112u) * 0x00800080u;  // 2^(sbyte-15) in both bf16 halves
  const uint32_t w[4] = {data.x, data.y, data.z, data.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t lo, hi;
    e4m3x4_to_bf16x2x2_scaled(w[k], lo, hi);
    out[2 * k] = bf16x2_mul(lo, c);
    out[2 * k + 1] = bf16x2_mul(hi, c);
  }
}

// 16 consecutive dims of an FP4 record: data = 8 bytes of e2m1 pairs (even
// dim in the low nibble), sbyte = the e4m3 scale of the 16-dim block.
// value = e2m1 * e4m3: at most 6 significant bits, in the f16 normal range,
// so the f16 product is exact and so is the bf16 result.
__device__ __forceinline__ void dequant_fp4_16(uint32_t lo_word, uint32_t hi_word, uint32_t sbyte,
                                               uint32_t (&out)[8]) {
  const uint32_t s16 = e4m3x2_to_f16x2(sbyte | (sbyte << 8));  // scale in both halves
  const uint32_t c = bf16x2_splat_pow2(112);
  const uint32_t w[2] = {lo_word, hi_word};
#pragma unroll
  for (int k = 0; k < 2; ++k) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t h = e2m1x2_to_f16x2((w[k] >> (8 * j)) & 0xFFu);
      uint32_t p;
      asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p) : "r"(h), "r"(s16));
      out[4 * k + j] = bf16x2_mul(f16x2_to_bf16x2_scaled(p), c);
    }
  }
}

// ---------------------------------------------------------------------------
// FP8 record encoding (the KV-cache writer and the FP8 output epilogue):
// per 32-value block the least power of two 2^e with amax * 2^-e <= 448
// (scale byte 127 + e; 0 for an all-zero block; e clamped to [-127, 127]),
// each value x * 2^-e rounded to the nearest E4M3FN, ties to even,
// saturating.  For fp32 inputs both steps are exact decisions: the scaling
// is by a power of two and the conversion rounds the exact value once.
// ---------------------------------------------------------------------------

// Two floats -> two E4M3FN bytes (lo in byte 0), nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Least e with amax * 2^-e <= 448 (0 for amax == 0), clamped to [-127, 127].
// Conjugate rotary embedding of one interleaved pair (a, b) by
// phi = pos * freq ("deepseek-ai/FlashMLA", "What it is": the output-side
// RoPE), in two steps so that a kernel can compute each pair's angle once
// and apply it to many rows: rope_cos_sin takes the angle in double,
// reduces it to [-pi, pi] (where the fast float sine and cosine are within
// 2^-21 absolute, far below one E4M3 step of the result) and returns its
// float cosine and sine; rope_conj_apply maps (a, b) -> (a cos + b sin,
// b cos - a sin), rounded in one fixed order so that every kernel using the
// pair of routines gives the same bytes.
__device__ __forceinline__ void rope_cos_sin(double pos, double freq, float& cs, float& sn) {
  double phi = pos * freq;
  phi -= 6.283185307179586 * rint(phi * 0.15915494309189535);
  __sincosf(static_cast<float>(phi), &sn, &cs);
}
__device__ __forceinline__ void rope_conj_apply(float& a, float& b, float cs, float sn) {
  const float x = a, y = b;
  a = __fmaf_rn(x, cs, __fmul_rn(y, sn));
  b = __fmaf_rn(y, cs, -__fmul_rn(x, sn));
}

__device__ __forceinline__ int fp8_block_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int E;
  frexpf(amax, &E);  // amax = f 2^E, f in [0.5, 1)
  int e = E - 10;    // amax 2^-e >= 2^9 > 448
  while (ldexpf(amax, -e) > 448.f) ++e;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

}  // namespace mla
