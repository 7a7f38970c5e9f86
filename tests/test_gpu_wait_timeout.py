"""Failure detection without a GPU fault: a bounded on-chip wait that nothing
ever satisfies gives up after its limit, ORs MLA_DEVERR_TIMEOUT into the
device error word and returns, and the context stays usable.

The kernel here is test-only: it is compiled from this file against the
library's own device helpers (mla_device.cuh: mbar_init, mbar_wait) and waits
on an mbarrier that nothing arrives on, with a 1 ms limit."""
import ctypes
import os
import subprocess

import pytest
import torch

import fp4_kv_cache_sparse_gb300 as mla
import synth
from fp4_kv_cache_sparse_gb300 import build as mla_build
from _harness import DeviceWorkload, all_queries, compare

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp4_kv_cache_sparse_gb300", "csrc")

SRC = r"""
#include <cstdint>
#include "mla_device.cuh"

__global__ void wait_for_nothing(int32_t* err, unsigned long long limit_ns) {
  __shared__ alignas(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mla::mbar_init(&bar, 1);
    abort_flag = 0;
  }
  __syncthreads();
  // No thread ever arrives, so phase 0 never completes.
  mla::mbar_wait(&bar, 0, &abort_flag, err, limit_ns);
}

extern "C" int wait_for_nothing_launch(int32_t* err, unsigned long long limit_ns) {
  wait_for_nothing<<<1, 32>>>(err, limit_ns);
  return static_cast<int>(cudaDeviceSynchronize());
}
"""


@pytest.fixture(scope="module")
def waitlib(tmp_path_factory):
    d = tmp_path_factory.mktemp("waitlib")
    src, so = d / "wait.cu", d / "libwait.so"
    src.write_text(SRC)
    subprocess.check_call([mla_build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                           "-shared", "-Xcompiler", "-fPIC", "-I", CSRC, "-o", str(so), str(src)])
    lib = ctypes.CDLL(str(so))
    lib.wait_for_nothing_launch.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong]
    lib.wait_for_nothing_launch.restype = ctypes.c_int
    return lib


def test_unsatisfied_wait_times_out_and_flags(waitlib):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = waitlib.wait_for_nothing_launch(err.data_ptr(), 1_000_000)  # 1 ms
    assert rc == 0  # the kernel returned: no fault, no hang
    assert int(err.item()) & mla.DEVERR_TIMEOUT
    # The context is still usable: a decode afterwards is correct and clean.
    w = synth.make_workload(0, workers=1)
    out, lse, e = DeviceWorkload(w).run()
    assert e == 0
    compare(out, lse, w, all_queries(w))
