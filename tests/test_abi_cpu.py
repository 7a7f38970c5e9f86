"""The C-ABI library without a GPU: it loads, exports every function
include/mla.h declares, and its host-side validation and planning answer
without touching the device (every call here fails validation or runs in
query mode, so nothing is launched)."""
import ctypes
import math
import os
import re

import pytest

from conftest import ROOT

import fp4_kv_cache_sparse_gb300 as mla
from fp4_kv_cache_sparse_gb300 import build as lib_build

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return mla.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(mla_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"mla_get_metadata", "mla_sparse_decode", "mla_combine", "mla_dequantize",
            "mla_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    # and nothing in the header is a torch type
    assert "torch" not in open(os.path.join(ROOT, "include", "mla.h")).read().lower()


def test_problem_struct_layout_matches_header():
    assert ctypes.sizeof(mla.Problem) == 64
    assert mla.Problem.num_pages.offset == 32 and mla.Problem.sm_scale.offset == 60


def _prob(**kw):
    base = dict(batch=2, seq_len_q=1, h_q=64, topk=300, num_pages=20)
    base.update(kw)
    return mla.Problem.make(**base)


def _query(lib, p, num_sms=152):
    parts = ctypes.c_int32(-1)
    ws = ctypes.c_size_t(0)
    st = lib.mla_get_metadata(ctypes.byref(p), num_sms, None, None, ctypes.byref(parts), ctypes.byref(ws), None)
    return st, parts.value, ws.value


def test_status_strings(lib):
    for s in range(6):
        assert lib.mla_status_string(s)
    assert lib.mla_status_string(0) == b"ok"


@pytest.mark.parametrize("kw,status", [
    (dict(kv_format=mla.KV_FP4_288), UNSUPPORTED),                 # FP4 only as the extra cache
    (dict(kv_format=mla.KV_BF16), UNSUPPORTED),                    # no bf16 KV in decode
    (dict(kv_format=mla.KV_NONE), INVALID),
    (dict(head_dim=576), UNSUPPORTED),
    (dict(page_size=32), UNSUPPORTED),
    (dict(num_kv_heads=2), UNSUPPORTED),
    (dict(h_q=48), UNSUPPORTED),
    (dict(h_q=256), UNSUPPORTED),
    (dict(batch=0), INVALID),
    (dict(topk=0), INVALID),
    (dict(num_pages=0), INVALID),
    (dict(sm_scale=float("nan")), INVALID),
    (dict(extra_topk=64, extra_num_pages=4, extra_kv_format=mla.KV_FP8_528), UNSUPPORTED),
    (dict(extra_topk=64, extra_num_pages=4, extra_kv_format=mla.KV_BF16), UNSUPPORTED),
    (dict(extra_topk=64, extra_num_pages=0), INVALID),
])
def test_problem_validation(lib, kw, status):
    st, _, _ = _query(lib, _prob(**kw))
    assert st == status


def _plan(p, num_sms):
    """Restatement of the partition rule: items = query tokens x tiles of
    128 slots; about num_sms / head_groups parts of equal size."""
    nh = min(p.h_q, 64)
    n_hg = p.h_q // nh
    T = math.ceil(p.topk / 128) + math.ceil(p.extra_topk / 128)
    nq = p.batch * p.seq_len_q
    G = nq * T
    target = min(max(num_sms // n_hg, 1), G)
    S = math.ceil(G / target)
    parts = math.ceil(G / S)
    max_splits = nq + parts
    ws_o = max_splits * p.h_q * 512 * 4
    ws_o = (ws_o + 255) // 256 * 256
    return parts, ws_o + max_splits * p.h_q * 4


@pytest.mark.parametrize("shape", [
    dict(batch=1, seq_len_q=1, h_q=16, topk=64, num_pages=2),
    dict(batch=64, seq_len_q=1, h_q=64, topk=2048, num_pages=64 * 512),
    dict(batch=128, seq_len_q=2, h_q=128, topk=2048, num_pages=128 * 2048),
    dict(batch=64, seq_len_q=1, h_q=64, topk=2048, num_pages=64 * 1024, extra_topk=512, extra_num_pages=64 * 256),
    dict(batch=32, seq_len_q=1, h_q=16, topk=65536, num_pages=32 * 16384),
    dict(batch=3, seq_len_q=2, h_q=32, topk=200, num_pages=50),
])
@pytest.mark.parametrize("num_sms", [1, 7, 152, 1000])
def test_metadata_query_mode(lib, shape, num_sms):
    p = mla.Problem.make(**shape)
    st, parts, ws = _query(lib, p, num_sms)
    assert st == OK
    assert (parts, ws) == _plan(p, num_sms)


def test_decode_argument_checks_before_any_launch(lib):
    p = _prob()
    st, parts, ws = _query(lib, p)
    A = ctypes.c_void_p(1 << 20)           # aligned fake device addresses: never dereferenced
    mis = ctypes.c_void_p((1 << 20) + 8)

    def call(q=A, kv=A, idx=A, xkv=None, xidx=None, sched=A, nsp=A, nparts=parts, wsp=A, wsb=ws,
             out=A, lse=A, prob=p):
        return lib.mla_sparse_decode(ctypes.byref(prob), q, kv, idx, xkv, xidx, sched, nsp, nparts, wsp, wsb,
                                     out, lse, None, None)

    assert call(q=None) == INVALID
    assert call(kv=None) == INVALID
    assert call(idx=None) == INVALID
    assert call(out=None) == INVALID
    assert call(q=mis) == INVALID                   # 16-byte alignment of q
    assert call(kv=mis) == INVALID                  # and of the record pool
    assert call(wsb=ws - 1) == WORKSPACE
    assert call(wsp=None) == WORKSPACE
    assert call(nparts=0) == INVALID
    px = _prob(extra_topk=100, extra_num_pages=3)
    _, parts_x, ws_x = _query(lib, px)
    assert call(prob=px, nparts=parts_x, wsb=ws_x) == INVALID    # extra cache missing
    assert call(prob=_prob(kv_format=mla.KV_FP4_288)) == UNSUPPORTED


def test_combine_and_dequantize_argument_checks(lib):
    p = _prob()
    A = ctypes.c_void_p(1 << 20)
    assert lib.mla_combine(ctypes.byref(p), None, A, A, A, A, None) == INVALID
    assert lib.mla_dequantize(mla.KV_BF16, A, 4, A, None) == UNSUPPORTED
    assert lib.mla_dequantize(7, A, 4, A, None) == INVALID
    assert lib.mla_dequantize(mla.KV_FP8_528, ctypes.c_void_p((1 << 20) + 4), 4, A, None) == INVALID
    assert lib.mla_dequantize(mla.KV_FP8_528, A, -1, A, None) == INVALID


def test_kv_write_argument_checks(lib):
    """Validation before any launch (no GPU needed): formats, sizes,
    pointers, alignment; n = 0 is a no-op."""
    A = ctypes.c_void_p(1 << 20)
    I = ctypes.c_void_p((1 << 20) + 64)
    assert lib.mla_kv_write(mla.KV_BF16, A, I, 4, A, 8, None, None) == UNSUPPORTED
    assert lib.mla_kv_write(0, A, I, 4, A, 8, None, None) == INVALID
    assert lib.mla_kv_write(mla.KV_FP8_528, A, I, -1, A, 8, None, None) == INVALID
    assert lib.mla_kv_write(mla.KV_FP8_528, A, I, 4, A, -1, None, None) == INVALID
    assert lib.mla_kv_write(mla.KV_FP8_528, None, I, 4, A, 8, None, None) == INVALID
    assert lib.mla_kv_write(mla.KV_FP4_288, A, None, 4, A, 8, None, None) == INVALID
    assert lib.mla_kv_write(mla.KV_FP8_528, ctypes.c_void_p((1 << 20) + 8), I, 4, A, 8, None, None) == INVALID
    assert lib.mla_kv_write(mla.KV_FP8_528, A, ctypes.c_void_p((1 << 20) + 2), 4, A, 8, None, None) == INVALID
    assert lib.mla_kv_write(mla.KV_FP8_528, A, I, 0, A, 8, None, None) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        mla.dequantize(torch.zeros((4, 528), dtype=torch.uint8))


def test_rope_fp8_decode_argument_checks_before_any_launch(lib):
    """The fused-epilogue decode validates the problem first, then its own
    arguments (positions, theta, the FP8 output), before any launch."""
    p = _prob()
    st, parts, ws = _query(lib, p)
    A = ctypes.c_void_p(1 << 20)

    def call(pos=A, theta=10000.0, out=A, prob=p, lse=A):
        return lib.mla_sparse_decode_rope_fp8(ctypes.byref(prob), A, A, A, None, None, A, A, parts, A, ws, pos,
                                              ctypes.c_float(theta), out, lse, None, None)

    assert call(pos=None) == INVALID
    assert call(pos=ctypes.c_void_p((1 << 20) + 2)) == INVALID
    assert call(out=None) == INVALID
    assert call(theta=1.0) == INVALID
    assert call(theta=float("nan")) == INVALID
    assert call(theta=float("inf")) == INVALID
    assert call(lse=None) == INVALID
    assert call(prob=_prob(h_q=48), pos=None) == UNSUPPORTED       # the problem is checked first
