// api.cu -- the C ABI (include/mla.h): argument validation, work planning
// and kernel launches.  No allocation, no host synchronisation.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mla.h"
#include "mla_internal.h"

namespace mla {

// Shape checks shared by every entry point.
mla_status_t validate_problem(const mla_problem_t* p) {
  if (p == nullptr) return MLA_ERR_INVALID_ARG;
  if (p->batch < 1 || p->seq_len_q < 1 || p->topk < 1 || p->extra_topk < 0 || p->h_q < 1) return MLA_ERR_INVALID_ARG;
  if (p->num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(p->sm_scale)) return MLA_ERR_INVALID_ARG;
  // The record format decides the kernel: FP4 only as the extra cache, no bf16 cache.
  if (p->kv_format == MLA_KV_FP4_288 || p->kv_format == MLA_KV_BF16) return MLA_ERR_UNSUPPORTED;
  if (p->kv_format != MLA_KV_FP8_528) return MLA_ERR_INVALID_ARG;
  if (p->head_dim != MLA_HEAD_DIM || p->page_size != MLA_PAGE_SIZE || p->num_kv_heads != 1)
    return MLA_ERR_UNSUPPORTED;
  if (!(p->h_q == 16 || p->h_q == 32 || p->h_q == 64 || p->h_q == 128)) return MLA_ERR_UNSUPPORTED;
  if (p->extra_topk > 0) {
    if (p->extra_kv_format == MLA_KV_BF16 || p->extra_kv_format == MLA_KV_FP8_528) return MLA_ERR_UNSUPPORTED;
    if (p->extra_kv_format != MLA_KV_FP4_288) return MLA_ERR_INVALID_ARG;
    if (p->extra_num_pages < 1) return MLA_ERR_INVALID_ARG;
  }
  const int64_t nq = static_cast<int64_t>(p->batch) * p->seq_len_q;
  const int64_t T = (p->topk + 127) / 128 + (static_cast<int64_t>(p->extra_topk) + 127) / 128;
  if (nq * T >= (int64_t(1) << 31) || nq * p->h_q >= (int64_t(1) << 31)) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

// Shape part of the plan plus the workspace layout for a given part count.
Plan plan_for_parts(const mla_problem_t* p, int num_parts) {
  Plan pl{};
  pl.nh = p->h_q < 64 ? p->h_q : 64;
  pl.n_hg = p->h_q / pl.nh;
  pl.Tm = (p->topk + 127) / 128;
  pl.Te = (p->extra_topk + 127) / 128;
  pl.T = pl.Tm + pl.Te;
  const int64_t nq = static_cast<int64_t>(p->batch) * p->seq_len_q;
  pl.G = nq * pl.T;
  pl.num_parts = num_parts;
  pl.S = num_parts > 0 ? (pl.G + num_parts - 1) / num_parts : 0;
  pl.max_splits = nq + num_parts;
  pl.ws_o_bytes = static_cast<size_t>(pl.max_splits) * p->h_q * MLA_HEAD_DIM * sizeof(float);
  pl.ws_o_bytes = (pl.ws_o_bytes + 255) & ~size_t(255);
  pl.ws_bytes = pl.ws_o_bytes + static_cast<size_t>(pl.max_splits) * p->h_q * sizeof(float);
  return pl;
}

namespace {

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
std::mutex g_sm_mutex;

mla_status_t device_sm_count(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices) {
    std::lock_guard<std::mutex> lock(g_sm_mutex);
    if (g_sm_count[dev] == 0) {
      int n = 0;
      if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;
      g_sm_count[dev] = n;
    }
    *out = g_sm_count[dev];
    return MLA_OK;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;
  *out = n;
  return MLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Balanced partition: about one part per SM for each head group (a CTA
// fills an SM), never more parts than work items.
Plan make_plan(const mla_problem_t* p, int num_sms) {
  Plan pl = plan_for_parts(p, 1);
  int64_t target = num_sms / pl.n_hg;
  if (target < 1) target = 1;
  if (target > pl.G) target = pl.G;
  const int64_t S = (pl.G + target - 1) / target;
  pl = plan_for_parts(p, static_cast<int>((pl.G + S - 1) / S));
  pl.S = S;
  return pl;
}

// The 128-head cluster kernel runs 128-head problems without an extra
// cache; every other shape runs on the swap-AB kernel.
bool uses_pair_kernel(const mla_problem_t* problem) { return problem->h_q == 128 && problem->extra_topk == 0; }

// Where the decode kernels write the fused epilogue's FP8 records of query
// tokens that have one split.
struct RopeOut {
  uint8_t* out;
  const int32_t* positions;
  RopeFreqs freqs;
};

}  // namespace

// Validation and the decode kernel's launch, shared by the bf16 and the
// FP8 output calls.  With rope, query tokens of one split are written as FP8
// records there instead of to out (which may then be null); *pout receives
// the parameters.
mla_status_t decode_launch(const mla_problem_t* problem, const void* q, const void* kv, const int32_t* indices,
                           const void* extra_kv, const int32_t* extra_indices, const int32_t* d_sched,
                           const int32_t* d_num_splits, int32_t num_parts, void* workspace, size_t workspace_bytes,
                           uint16_t* out, float* lse, int32_t* d_error, const RopeOut* rope, mla_stream_t stream,
                           DecodeParams* pout) {
  mla_status_t st = validate_problem(problem);
  if (st != MLA_OK) return st;
  if (q == nullptr || kv == nullptr || indices == nullptr || d_sched == nullptr || d_num_splits == nullptr ||
      lse == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(indices) & 3u))
    return MLA_ERR_INVALID_ARG;
  if (problem->extra_topk > 0) {
    if (extra_kv == nullptr || extra_indices == nullptr || !aligned16(extra_kv) ||
        (reinterpret_cast<uintptr_t>(extra_indices) & 3u))
      return MLA_ERR_INVALID_ARG;
  }
  // The part ranges live in d_sched (checked on the device); the host needs
  // only the part count for the grid and the workspace layout.
  Plan pl = plan_for_parts(problem, num_parts);
  if (num_parts < 1 || num_parts > pl.G) return MLA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < pl.ws_bytes) return MLA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int nq = problem->batch * problem->seq_len_q;

  DecodeParams& p = *pout;
  p = DecodeParams{};
  p.q = static_cast<const uint16_t*>(q);
  p.kv = static_cast<const uint8_t*>(kv);
  p.idx = indices;
  p.xkv = problem->extra_topk > 0 ? static_cast<const uint8_t*>(extra_kv) : nullptr;
  p.xidx = problem->extra_topk > 0 ? extra_indices : nullptr;
  p.sched = d_sched;
  p.num_splits = d_num_splits;
  p.ws_o = static_cast<float*>(workspace);
  p.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.ws_o_bytes);
  p.ws_splits_cap = pl.max_splits;
  p.out = out;
  p.lse = lse;
  p.d_error = d_error;
  p.nq = nq;
  p.h_q = problem->h_q;
  p.n_hg = pl.n_hg;
  p.topk = problem->topk;
  p.xtopk = problem->extra_topk;
  p.Tm = pl.Tm;
  p.T = pl.T;
  const int64_t cap = int64_t(1) << 31;
  p.pool_tokens = problem->num_pages * MLA_PAGE_SIZE < cap ? problem->num_pages * MLA_PAGE_SIZE : cap;
  p.xpool_tokens = problem->extra_topk > 0
                       ? (problem->extra_num_pages * MLA_PAGE_SIZE < cap ? problem->extra_num_pages * MLA_PAGE_SIZE
                                                                          : cap)
                       : 0;
  p.scale_log2 = problem->sm_scale * 1.4426950408889634f;
  if (rope != nullptr) {
    p.rope_out = rope->out;
    p.positions = rope->positions;
    p.rope = rope->freqs;
  }

  const int grid = pl.num_parts * pl.n_hg;
  cudaError_t e;
  if (uses_pair_kernel(problem)) {
    // All 128 heads on the MMA's M dimension, the latent dims split over a
    // 2-CTA cluster (same part count and SM budget as two 64-head groups).
    e = launch_decode_pair(p, pl.num_parts, s);
  } else {
    switch (pl.nh) {
      case 64: e = launch_decode<64>(p, grid, s); break;
      case 32: e = launch_decode<32>(p, grid, s); break;
      default: e = launch_decode<16>(p, grid, s); break;
    }
  }
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported problem";
    case MLA_ERR_WORKSPACE: return "workspace too small";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_TIMEOUT: return "timeout";
  }
  return "unknown status";
}

mla_status_t mla_get_metadata(const mla_problem_t* problem, int32_t num_sms, int32_t* d_sched,
                              int32_t* d_num_splits, int32_t* num_parts_out, size_t* workspace_bytes_out,
                              mla_stream_t stream) {
  mla_status_t st = validate_problem(problem);
  if (st != MLA_OK) return st;
  if (num_parts_out == nullptr || workspace_bytes_out == nullptr || num_sms < 0) return MLA_ERR_INVALID_ARG;
  if ((d_sched == nullptr) != (d_num_splits == nullptr)) return MLA_ERR_INVALID_ARG;
  if (num_sms == 0) {
    st = device_sm_count(&num_sms);
    if (st != MLA_OK) return st;
  }
  const Plan pl = make_plan(problem, num_sms);
  *num_parts_out = pl.num_parts;
  *workspace_bytes_out = pl.ws_bytes;
  if (d_sched == nullptr) return MLA_OK;
  const int nq = problem->batch * problem->seq_len_q;
  if (launch_metadata(pl, nq, d_sched, d_num_splits, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_sparse_decode(const mla_problem_t* problem, const void* q, const void* kv, const int32_t* indices,
                               const void* extra_kv, const int32_t* extra_indices, const int32_t* d_sched,
                               const int32_t* d_num_splits, int32_t num_parts, void* workspace,
                               size_t workspace_bytes, void* out, float* lse, int32_t* d_error,
                               mla_stream_t stream) {
  mla_status_t st = validate_problem(problem);
  if (st != MLA_OK) return st;
  if (out == nullptr || !aligned16(out)) return MLA_ERR_INVALID_ARG;
  DecodeParams p{};
  st = decode_launch(problem, q, kv, indices, extra_kv, extra_indices, d_sched, d_num_splits, num_parts, workspace,
                     workspace_bytes, static_cast<uint16_t*>(out), lse, d_error, nullptr, stream, &p);
  if (st != MLA_OK) return st;
  if (num_parts > 1) {
    // Only query tokens with more than one split have partials to merge: a
    // grid over parts visits just those (at most one per part) and is the
    // smaller grid when parts are fewer than query tokens; otherwise one warp
    // per row, the kernel skipping one-split rows.
    const int32_t* by_part = num_parts < p.nq ? d_sched : nullptr;
    if (launch_combine(d_num_splits, p.ws_o, p.ws_lse, p.out, lse, p.nq, problem->h_q, true, by_part, num_parts,
                       p.T, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status_t mla_sparse_decode_rope_fp8(const mla_problem_t* problem, const void* q, const void* kv,
                                        const int32_t* indices, const void* extra_kv, const int32_t* extra_indices,
                                        const int32_t* d_sched, const int32_t* d_num_splits, int32_t num_parts,
                                        void* workspace, size_t workspace_bytes, const int32_t* positions,
                                        float rope_theta, void* out_fp8, float* lse, int32_t* d_error,
                                        mla_stream_t stream) {
  mla_status_t st = validate_problem(problem);
  if (st != MLA_OK) return st;
  if (out_fp8 == nullptr || positions == nullptr || (reinterpret_cast<uintptr_t>(positions) & 3u) ||
      (reinterpret_cast<uintptr_t>(out_fp8) & 3u))
    return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(rope_theta) || !(rope_theta > 1.f)) return MLA_ERR_INVALID_ARG;
  RopeOut ro{};
  ro.out = static_cast<uint8_t*>(out_fp8);
  ro.positions = positions;
  for (int j = 0; j < 32; ++j) ro.freqs.f[j] = std::pow(static_cast<double>(rope_theta), -2.0 * j / 64.0);
  // The decode kernels write the records of one-split query tokens
  // themselves; only split tokens go through the workspace to the merge.
  DecodeParams p{};
  st = decode_launch(problem, q, kv, indices, extra_kv, extra_indices, d_sched, d_num_splits, num_parts, workspace,
                     workspace_bytes, nullptr, lse, d_error, &ro, stream, &p);
  if (st != MLA_OK) return st;
  if (launch_rope_fp8(d_num_splits, p.ws_o, p.ws_lse, positions, ro.freqs, ro.out, lse, p.nq, problem->h_q, true,
                      num_parts < p.nq ? d_sched : nullptr, num_parts, p.T,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_combine(const mla_problem_t* problem, const int32_t* d_num_splits, const float* o_partial,
                         const float* lse_partial, void* out, float* lse, mla_stream_t stream) {
  mla_status_t st = validate_problem(problem);
  if (st != MLA_OK) return st;
  if (d_num_splits == nullptr || o_partial == nullptr || lse_partial == nullptr || out == nullptr || lse == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_partial) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse_partial) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_ERR_INVALID_ARG;
  const int nq = problem->batch * problem->seq_len_q;
  if (launch_combine(d_num_splits, o_partial, lse_partial, static_cast<uint16_t*>(out), lse, nq, problem->h_q,
                     false, nullptr, 0, 0, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_dequantize(int32_t kv_format, const void* records, int64_t n, void* out, mla_stream_t stream) {
  if (kv_format != MLA_KV_FP8_528 && kv_format != MLA_KV_FP4_288) {
    return kv_format == MLA_KV_BF16 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  }
  if (n < 0 || (n > 0 && (records == nullptr || out == nullptr))) return MLA_ERR_INVALID_ARG;
  if (n > 0 && (!aligned16(records) || !aligned16(out))) return MLA_ERR_INVALID_ARG;
  if (n * 32 >= (int64_t(1) << 40)) return MLA_ERR_UNSUPPORTED;
  if (launch_dequant(kv_format, static_cast<const uint8_t*>(records), n, static_cast<uint16_t*>(out),
                     reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_kv_write(int32_t kv_format, const void* latents, const int32_t* slots, int64_t n, void* pool,
                          int64_t num_pages, int32_t* d_error, mla_stream_t stream) {
  if (kv_format != MLA_KV_FP8_528 && kv_format != MLA_KV_FP4_288) {
    return kv_format == MLA_KV_BF16 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  }
  if (n < 0 || num_pages < 0) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (latents == nullptr || slots == nullptr || pool == nullptr) return MLA_ERR_INVALID_ARG;
  if (!aligned16(latents) || !aligned16(pool) || (reinterpret_cast<uintptr_t>(slots) & 3u) != 0)
    return MLA_ERR_INVALID_ARG;
  if (n * MLA_HEAD_DIM >= (int64_t(1) << 40)) return MLA_ERR_UNSUPPORTED;
  const int64_t cap = int64_t(1) << 31;
  const int64_t pool_tokens = num_pages * MLA_PAGE_SIZE < cap ? num_pages * MLA_PAGE_SIZE : cap;
  if (launch_kv_write(kv_format, static_cast<const uint16_t*>(latents), slots, n, static_cast<uint8_t*>(pool),
                      pool_tokens, d_error, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // extern "C"
