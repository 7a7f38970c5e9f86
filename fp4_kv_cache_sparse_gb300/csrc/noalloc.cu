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
// a device address, so every call looks the address up with
// cudaGetSymbolAddress on the current device and passes it on.  Looking it
// up per call (a host-side query) keeps the address right even after a
// device reset has rebuilt the context; the first lookup on a device also
// loads this library's device code there, so that first call should come
// before any stream capture.  Every call then runs the ordinary
// mla_sparse_decode with that address as workspace.  The decode writes
// every partial it later reads, so nothing needs clearing between calls;
// calls that overlap on the GPU (other streams, other host threads) share
// the one array and race.
#include <cstdint>

#include "../../include/mla.h"
#include "mla_internal.h"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[MLA_NOALLOC_SCRATCH_BYTES];

}  // namespace

extern "C" mla_status_t mla_sparse_decode_noalloc(const mla_problem_t* problem, const void* q, const void* kv,
                                                  const int32_t* indices, const void* extra_kv,
                                                  const int32_t* extra_indices, const int32_t* d_sched,
                                                  const int32_t* d_num_splits, int32_t num_parts, void* out,
                                                  float* lse, int32_t* d_error, mla_stream_t stream) {
  // The problem is checked first, so an invalid or unsupported problem gets
  // that status and not MLA_ERR_WORKSPACE.
  const mla_status_t st = mla::validate_problem(problem);
  if (st != MLA_OK) return st;
  if (num_parts < 1) return MLA_ERR_INVALID_ARG;
  // The same workspace size mla_get_metadata reports for this part count.
  if (mla::plan_for_parts(problem, num_parts).ws_bytes > MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_decode_scratch) != cudaSuccess || scratch == nullptr) return MLA_ERR_CUDA;
  return mla_sparse_decode(problem, q, kv, indices, extra_kv, extra_indices, d_sched, d_num_splits, num_parts,
                           scratch, MLA_NOALLOC_SCRATCH_BYTES, out, lse, d_error, stream);
}
