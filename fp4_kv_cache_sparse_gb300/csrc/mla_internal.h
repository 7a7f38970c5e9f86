// mla_internal.h -- host/device interface between the C-ABI layer and the
// kernels of the library (not installed, not part of the ABI).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mla.h"

namespace mla {

// Everything the decode kernel reads, resolved by the host layer.
// Output-side rotary frequencies of the fused epilogue: freqs[j] =
// theta^(-2j/64) for the pair (448 + 2j, 449 + 2j).
struct RopeFreqs {
  double f[32];
};

struct DecodeParams {
  const uint16_t* q;        // bf16 [nq][h_q][512]
  const uint8_t* kv;        // FP8 records
  const int32_t* idx;       // [nq][topk]
  const uint8_t* xkv;       // FP4 records (extra cache) or null
  const int32_t* xidx;      // [nq][xtopk] or null
  const int32_t* sched;     // [num_parts][8]
  const int32_t* num_splits;  // [nq + 1]
  float* ws_o;              // [ws_splits_cap][h_q][512]
  float* ws_lse;            // [ws_splits_cap][h_q]
  int64_t ws_splits_cap;
  uint16_t* out;            // bf16 [nq][h_q][512]
  float* lse;               // [nq][h_q]
  int32_t* d_error;         // nullable
  int nq, h_q, n_hg, topk, xtopk, Tm, T;
  int64_t pool_tokens, xpool_tokens;
  float scale_log2;         // sm_scale * log2(e)
  // Fused output epilogue written by the decode kernel itself for query
  // tokens of one split: null, or [nq][h_q][528] FP8 records after the
  // conjugate rotary embedding at positions[qidx].
  uint8_t* rope_out;
  const int32_t* positions;
  RopeFreqs rope;
};

// Work plan derived from the problem shape and the SM count.
struct Plan {
  int nh;          // heads per CTA (16, 32 or 64)
  int n_hg;        // head groups = h_q / nh
  int Tm, Te, T;   // tiles per query token: main, extra, total
  int64_t G;       // total (query token, tile) items
  int64_t S;       // items per part
  int num_parts;
  int64_t max_splits;
  size_t ws_o_bytes, ws_bytes;
};

// Shape checks shared by every entry point (MLA_OK or the status to return).
mla_status_t validate_problem(const mla_problem_t* p);

// Shape part of the plan plus the workspace layout (ws_bytes) for a given
// part count; the one definition of the workspace size.
Plan plan_for_parts(const mla_problem_t* p, int num_parts);

template <int NH>
cudaError_t launch_decode(const DecodeParams& p, int grid, cudaStream_t stream);
int decode_smem_bytes(int nh);

// 128 heads, FP8 main cache only: a 2-CTA cluster per part splitting the latent dims.
cudaError_t launch_decode_pair(const DecodeParams& p, int num_parts, cudaStream_t stream);
int decode_pair_smem_bytes();

cudaError_t launch_metadata(const Plan& plan, int nq, int32_t* d_sched, int32_t* d_num_splits, cudaStream_t stream);

// Merge of split partials.  With sched (the decode's part schedule, T
// tiles per query token) only the rows of query tokens that have several
// splits are visited, every other row having been written by the decode
// kernel; without it every row is (skip_single then skips one-split rows).
cudaError_t launch_combine(const int32_t* d_num_splits, const float* o_part, const float* lse_part, uint16_t* out,
                           float* lse, int nq, int h_q, bool skip_single, const int32_t* sched, int num_parts, int T,
                           cudaStream_t stream);

// Merge of each query token's split partials (with skip_single, only tokens
// of more than one split), conjugate rotary embedding of dims 448..511 and
// the cast to 528-byte FP8 records.
cudaError_t launch_rope_fp8(const int32_t* d_num_splits, const float* o_part, const float* lse_part,
                            const int32_t* positions, const RopeFreqs& freqs, uint8_t* out, float* lse, int nq,
                            int h_q, bool skip_single, const int32_t* sched, int num_parts, int T,
                            cudaStream_t stream);

cudaError_t launch_dequant(int kv_format, const uint8_t* records, int64_t n, uint16_t* out, cudaStream_t stream);

cudaError_t launch_kv_write(int kv_format, const uint16_t* latents, const int32_t* slots, int64_t n, uint8_t* pool,
                            int64_t pool_tokens, int32_t* d_error, cudaStream_t stream);

// cuTensorMapEncodeTiled from the driver, looked up once (thread-safe
// static initialization); nullptr if the driver does not offer it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
inline EncodeTiledFn tensor_map_encoder() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    const bool ok = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                        cudaSuccess &&
                    q == cudaDriverEntryPointSuccess;
    return ok ? reinterpret_cast<EncodeTiledFn>(f) : EncodeTiledFn{nullptr};
  }();
  return fn;
}

// A kernel's dynamic shared memory limit, set once per device: the attribute
// belongs to the current device's context, so bit d of `done` records device
// d (devices past 63 set it on every call).
inline cudaError_t max_dynamic_smem_once(std::atomic<uint64_t>& done, const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace mla
