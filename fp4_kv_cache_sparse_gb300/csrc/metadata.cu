// metadata.cu -- tile-scheduler metadata ("flops/flashmla-decode-fp8-fp4-kv",
// "Workarounds": computed once before the decode loop; split decoding with
// num_splits).
//
// The work list is every (query token, tile) pair in query-major order,
// item g = qidx * T + t.  Part p owns items [p*S, min((p+1)*S, G)).  A query
// token cut by part boundaries becomes several splits; its split count and
// the local split id of a part's first query token follow from the same
// arithmetic, so the kernel is closed-form plus one prefix sum.
#include <cstdint>

#include "../../include/mla.h"
#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) metadata_kernel(int64_t G, int64_t S, int T, int num_parts, int nq,
                                                                int32_t* sched, int32_t* num_splits) {
  __shared__ int64_t partial[kScanThreads];
  const int tid = threadIdx.x;
  for (int p = tid; p < num_parts; p += kScanThreads) {
    const int64_t g0 = static_cast<int64_t>(p) * S;
    const int64_t g1 = min(G, g0 + S);
    const int64_t q0 = g0 / T;
    const int64_t first_part_of_q0 = (q0 * T) / S;
    int32_t* e = sched + static_cast<int64_t>(p) * MLA_SCHED_INTS;
    e[0] = static_cast<int32_t>(g0);
    e[1] = static_cast<int32_t>(g1);
    e[2] = static_cast<int32_t>(p - first_part_of_q0);
    e[3] = static_cast<int32_t>(q0);
    e[4] = e[5] = e[6] = e[7] = 0;
  }
  // splits(q) = (last part touching q) - (first part touching q) + 1
  const int per = (nq + kScanThreads - 1) / kScanThreads;
  const int qa = min(nq, tid * per), qb = min(nq, qa + per);
  int64_t local = 0;
  for (int q = qa; q < qb; ++q) {
    const int64_t first = (static_cast<int64_t>(q) * T) / S;
    const int64_t last = (static_cast<int64_t>(q + 1) * T - 1) / S;
    local += last - first + 1;
  }
  partial[tid] = local;
  __syncthreads();
  for (int off = 1; off < kScanThreads; off <<= 1) {  // inclusive scan
    const int64_t v = tid >= off ? partial[tid - off] : 0;
    __syncthreads();
    partial[tid] += v;
    __syncthreads();
  }
  int64_t run = partial[tid] - local;  // exclusive prefix of this thread's block
  for (int q = qa; q < qb; ++q) {
    num_splits[q] = static_cast<int32_t>(run);
    const int64_t first = (static_cast<int64_t>(q) * T) / S;
    const int64_t last = (static_cast<int64_t>(q + 1) * T - 1) / S;
    run += last - first + 1;
  }
  if (tid == kScanThreads - 1) num_splits[nq] = static_cast<int32_t>(partial[tid]);
}

}  // namespace

cudaError_t launch_metadata(const Plan& plan, int nq, int32_t* d_sched, int32_t* d_num_splits, cudaStream_t stream) {
  metadata_kernel<<<1, kScanThreads, 0, stream>>>(plan.G, plan.S, plan.T, plan.num_parts, nq, d_sched, d_num_splits);
  return cudaGetLastError();
}

}  // namespace mla
