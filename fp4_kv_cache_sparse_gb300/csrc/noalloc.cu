// noalloc.cu -- mla_sparse_decode_noalloc: the decode step for callers that
// cannot allocate device memory when they call it.
//
// Who needs it: code that receives only its input and output buffers and is
// not allowed to allocate -- a plugin or kernel hook running inside another
// runtime that owns all device memory through its own pool, or a serving
// loop that has reserved every byte up front and may not call cudaMalloc
// (which can also synchronise the device) on its per-step path.  Such a
// caller cannot provide the split-KV workspace that mla_sparse_decode takes.
//
// How: the workspace is a file-scope __device__ array of fixed size that the
// CUDA runtime places on every device that loads this library (it stays
// there until the process exits).  Host code cannot use the array's name as
// a device address, so the first call on each device looks its address up
// with cudaGetSymbolAddress (with that device current) and keeps it; that
// first call should therefore come before any stream capture.  Every call
// then runs the ordinary mla_sparse_decode with that address as workspace.
// The decode writes every partial it later reads, so nothing needs clearing
// between calls; calls that overlap on the GPU (other streams, other host
// threads) share the one array and race.
#include <cstdint>
#include <mutex>

#include "../../include/mla.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_scratch[MLA_NOALLOC_SCRATCH_BYTES];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Same upper bound as the workspace mla_get_metadata reports: one slot per
// query token plus one per part, each h_q x (512 + 1) floats, the output
// block padded to 256 bytes.
size_t workspace_bytes(const mla_problem_t* p, int32_t num_parts) {
  const size_t splits = static_cast<size_t>(p->batch) * p->seq_len_q + static_cast<size_t>(num_parts);
  size_t o = splits * p->h_q * MLA_HEAD_DIM * sizeof(float);
  o = (o + 255) & ~size_t(255);
  return o + splits * p->h_q * sizeof(float);
}

}  // namespace

extern "C" mla_status_t mla_sparse_decode_noalloc(const mla_problem_t* problem, const void* q, const void* kv,
                                                  const int32_t* indices, const void* extra_kv,
                                                  const int32_t* extra_indices, const int32_t* d_sched,
                                                  const int32_t* d_num_splits, int32_t num_parts, void* out,
                                                  float* lse, int32_t* d_error, mla_stream_t stream) {
  if (problem == nullptr || num_parts < 1 || problem->batch < 1 || problem->seq_len_q < 1 || problem->h_q < 1)
    return MLA_ERR_INVALID_ARG;
  if (workspace_bytes(problem, num_parts) > MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_decode_scratch) != cudaSuccess || addr == nullptr) return MLA_ERR_CUDA;
      g_scratch_addr[dev] = addr;
    }
    scratch = g_scratch_addr[dev];
  }
  return mla_sparse_decode(problem, q, kv, indices, extra_kv, extra_indices, d_sched, d_num_splits, num_parts,
                           scratch, MLA_NOALLOC_SCRATCH_BYTES, out, lse, d_error, stream);
}
