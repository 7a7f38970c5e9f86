"""mla_sparse_decode_noalloc: the decode step for callers that cannot
allocate device memory (a plugin handed only its I/O buffers by a host
runtime, a serving loop whose memory is all pre-reserved by its own pool).
Its split partials live in the library's fixed device array instead of a
caller workspace.  Checked through the C ABI against mla_sparse_decode on
the same inputs, twice in a row (the array keeps the previous call's
contents), and against the fp64 oracle on sampled query tokens.  Collected
last so that a failure here leaves the rest of the suite already run."""
import ctypes

import numpy as np
import pytest
import torch

import fp4_kv_cache_sparse_gb300 as mla
import synth
from _harness import DeviceWorkload, OUT_ATOL, OUT_RTOL, LSE_ATOL, compare, sample_queries

pytestmark = pytest.mark.gpu

NOALLOC_MAX = 128 * 1024 * 1024


def _lib():
    lib = mla.load()
    P = ctypes.c_void_p
    lib.mla_sparse_decode_noalloc.argtypes = [ctypes.POINTER(mla.Problem), P, P, P, P, P, P, P, ctypes.c_int32,
                                              P, P, P, P]
    lib.mla_sparse_decode_noalloc.restype = ctypes.c_int
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, dw, dec, out, lse, err):
    st = lib.mla_sparse_decode_noalloc(ctypes.byref(dw.problem), _p(dw.q), _p(dw.kv), _p(dw.idx), _p(dw.xkv),
                                       _p(dw.xidx), _p(dec.sched), _p(dec.num_splits), dec.num_parts,
                                       _p(out), _p(lse), _p(err),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _close(a_out, a_lse, b_out, b_lse):
    x, y = a_out.float(), b_out.float()
    assert torch.all((x - y).abs() <= OUT_ATOL + OUT_RTOL * y.abs())
    both = torch.isneginf(a_lse) & torch.isneginf(b_lse)
    assert torch.all(both | ((a_lse - b_lse).abs() <= LSE_ATOL))


@pytest.mark.parametrize("cid", [1, 2, 3])
def test_noalloc_matches_workspace_entry_point_twice(cid):
    """64 heads (FP8, and FP8 + FP4 extra cache) and 128 heads with two query
    tokens per sequence (the 2-CTA kernel and the merge)."""
    lib = _lib()
    w = synth.make_workload(cid, batch=8 if cid != 2 else 4, workers=1)
    dw = DeviceWorkload(w)
    dec = dw.decoder()
    assert dec.num_parts > 1 and dec.ws_bytes <= NOALLOC_MAX     # split partials are used
    ref_out, ref_lse = dec(dw.q, dw.kv, dw.idx, dw.xkv, dw.xidx)
    torch.cuda.synchronize()
    err = torch.zeros((1,), dtype=torch.int32, device=dw.dev)
    qs, oracle_ref = sample_queries(w, n=3, seed=cid), None
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _noalloc(lib, dw, dec, out, lse, err) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        _close(out, lse, ref_out, ref_lse)
        oracle_ref = compare(out, lse, w, qs, oracle_ref)


def test_noalloc_rejects_problems_beyond_its_array():
    lib = _lib()
    # 256 query tokens x 128 heads need ~87 MB of partials per 76 parts;
    # 4096 query tokens do not fit in the fixed array.
    p = mla.Problem.make(4096, 1, 128, 2048, 1 << 20)
    dev = torch.device("cuda", 0)
    dummy = torch.zeros((16,), dtype=torch.int32, device=dev)
    st = lib.mla_sparse_decode_noalloc(ctypes.byref(p), _p(dummy), _p(dummy), _p(dummy), None, None,
                                       _p(dummy), _p(dummy), 76, _p(dummy), _p(dummy), None, None)
    assert st == 3          # MLA_ERR_WORKSPACE, nothing enqueued


def test_noalloc_checks_the_problem_before_the_array_size():
    """An unsupported problem (48 heads) is reported as such, not as a
    workspace overflow, even when it would also overflow the array."""
    lib = _lib()
    p = mla.Problem.make(4096, 1, 48, 2048, 1 << 20)
    dev = torch.device("cuda", 0)
    dummy = torch.zeros((16,), dtype=torch.int32, device=dev)
    st = lib.mla_sparse_decode_noalloc(ctypes.byref(p), _p(dummy), _p(dummy), _p(dummy), None, None,
                                       _p(dummy), _p(dummy), 76, _p(dummy), _p(dummy), None, None)
    assert st == 2          # MLA_ERR_UNSUPPORTED, nothing enqueued
