"""fp64 CPU oracle for token-sparse MLA decode over a quantized paged KV cache.

TEST INFRASTRUCTURE ONLY.  Loaded by the test suite, by the smoke check and
by the CPU-baseline leg of the benchmark, never by the product path.  The
arithmetic lives in ``oracle.c`` (plain C, double precision, OpenMP over
heads); this module compiles it with gcc and marshals numpy arrays to it.  It
shares nothing with the GPU library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

D = 512
FP8_RECORD_BYTES = 528
FP4_RECORD_BYTES = 288


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-fno-fast-math", "-ffp-contract=off",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    lib.oracle_e4m3fn.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3fn.restype = ctypes.c_double
    lib.oracle_e8m0.argtypes = [ctypes.c_uint8]
    lib.oracle_e8m0.restype = ctypes.c_double
    lib.oracle_e2m1.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1.restype = ctypes.c_double
    lib.oracle_dequant_fp8.argtypes = [P, ctypes.c_longlong, P]
    lib.oracle_dequant_fp8.restype = None
    lib.oracle_dequant_fp4.argtypes = [P, ctypes.c_longlong, P]
    lib.oracle_dequant_fp4.restype = None
    lib.oracle_e4m3fn_rne.argtypes = [ctypes.c_double]
    lib.oracle_e4m3fn_rne.restype = ctypes.c_uint8
    lib.oracle_e2m1_rne.argtypes = [ctypes.c_double]
    lib.oracle_e2m1_rne.restype = ctypes.c_uint8
    lib.oracle_encode_fp8.argtypes = [P, ctypes.c_longlong, P]
    lib.oracle_encode_fp8.restype = None
    lib.oracle_encode_fp4.argtypes = [P, ctypes.c_longlong, P]
    lib.oracle_encode_fp4.restype = None
    lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
    lib.oracle_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_bf16_rne_array.argtypes = [P, ctypes.c_longlong, P]
    lib.oracle_bf16_rne_array.restype = None
    lib.oracle_sparse_mla_decode.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_longlong, ctypes.c_longlong, ctypes.c_float,
        P, P, P, P, P, P, P, P]
    lib.oracle_sparse_mla_decode.restype = ctypes.c_longlong
    lib.oracle_combine.argtypes = [ctypes.c_int, ctypes.c_longlong, P, P, P, P]
    lib.oracle_combine.restype = None
    lib.oracle_rope_rotate.argtypes = [P, ctypes.c_longlong, P, ctypes.c_double, ctypes.c_int]
    lib.oracle_rope_rotate.restype = None
    lib.oracle_rope_fp8_epilogue.argtypes = [P, ctypes.c_longlong, P, ctypes.c_double, P]
    lib.oracle_rope_fp8_epilogue.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e4m3fn(b: int) -> float:
    return _load().oracle_e4m3fn(b)


def e8m0(b: int) -> float:
    return _load().oracle_e8m0(b)


def e2m1(nib: int) -> float:
    return _load().oracle_e2m1(nib)


def dequant_fp8(records: np.ndarray) -> np.ndarray:
    """records: uint8 [n, 528] -> float64 [n, 512]."""
    r = np.ascontiguousarray(records, dtype=np.uint8).reshape(-1, FP8_RECORD_BYTES)
    out = np.empty((r.shape[0], D), dtype=np.float64)
    _load().oracle_dequant_fp8(_ptr(r), r.shape[0], _ptr(out))
    return out


def dequant_fp4(records: np.ndarray) -> np.ndarray:
    """records: uint8 [n, 288] -> float64 [n, 512]."""
    r = np.ascontiguousarray(records, dtype=np.uint8).reshape(-1, FP4_RECORD_BYTES)
    out = np.empty((r.shape[0], D), dtype=np.float64)
    _load().oracle_dequant_fp4(_ptr(r), r.shape[0], _ptr(out))
    return out


def e4m3fn_rne(x: float) -> int:
    """Nearest E4M3FN byte (ties to even, saturating at +-448)."""
    return int(_load().oracle_e4m3fn_rne(float(x)))


def e2m1_rne(x: float) -> int:
    """Nearest e2m1 nibble (ties to even, saturating at +-6)."""
    return int(_load().oracle_e2m1_rne(float(x)))


def encode_fp8(x: np.ndarray) -> np.ndarray:
    """float64 [n, 512] latents -> uint8 [n, 528] FP8 records (the writer's quantizer)."""
    x = np.ascontiguousarray(x, dtype=np.float64).reshape(-1, 512)
    out = np.empty((x.shape[0], 528), dtype=np.uint8)
    _load().oracle_encode_fp8(_ptr(x), x.shape[0], _ptr(out))
    return out


def encode_fp4(x: np.ndarray) -> np.ndarray:
    """float64 [n, 512] latents -> uint8 [n, 288] FP4 records (the writer's quantizer)."""
    x = np.ascontiguousarray(x, dtype=np.float64).reshape(-1, 512)
    out = np.empty((x.shape[0], 288), dtype=np.uint8)
    _load().oracle_encode_fp4(_ptr(x), x.shape[0], _ptr(out))
    return out


def bf16_rne(x) -> np.ndarray:
    """float64 array -> bfloat16 bit patterns (uint16), one RNE rounding."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_bf16_rne_array(_ptr(a), a.size, _ptr(out))
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def sparse_mla_decode(q_bits, kv, idx, sm_scale, extra_kv=None, extra_idx=None,
                      pool_tokens=None, extra_pool_tokens=None):
    """Run the oracle.

    q_bits: uint16 [b, s, h, 512] (bf16 patterns); kv: uint8 [pool, 528];
    idx: int32 [b, s, topk]; extra_kv: uint8 [xpool, 288]; extra_idx: int32
    [b, s, xtopk].  Returns dict(out_bf16, out_f64, lse, bad).
    """
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    b, s, h, d = q.shape
    assert d == D
    kv = np.ascontiguousarray(kv, dtype=np.uint8).reshape(-1, FP8_RECORD_BYTES)
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(b, s, -1)
    topk = idx.shape[2]
    if pool_tokens is None:
        pool_tokens = kv.shape[0]
    xtopk = 0
    if extra_idx is not None:
        extra_kv = np.ascontiguousarray(extra_kv, dtype=np.uint8).reshape(-1, FP4_RECORD_BYTES)
        extra_idx = np.ascontiguousarray(extra_idx, dtype=np.int32).reshape(b, s, -1)
        xtopk = extra_idx.shape[2]
        if extra_pool_tokens is None:
            extra_pool_tokens = extra_kv.shape[0]
    else:
        extra_kv = None
        extra_pool_tokens = 0
    out_bf16 = np.empty((b, s, h, D), dtype=np.uint16)
    out_f64 = np.empty((b, s, h, D), dtype=np.float64)
    lse = np.empty((b, s, h), dtype=np.float64)
    bad = _load().oracle_sparse_mla_decode(
        b, s, h, topk, xtopk, int(pool_tokens), int(extra_pool_tokens),
        ctypes.c_float(np.float32(sm_scale)),
        _ptr(q), _ptr(kv), _ptr(idx), _ptr(extra_kv), _ptr(extra_idx),
        _ptr(out_bf16), _ptr(out_f64), _ptr(lse))
    return dict(out_bf16=out_bf16, out_f64=out_f64, lse=lse, bad=int(bad))


def combine(o_part: np.ndarray, lse_part: np.ndarray):
    """o_part: float64 [n, rows, 512]; lse_part: float64 [n, rows]."""
    o = np.ascontiguousarray(o_part, dtype=np.float64)
    l = np.ascontiguousarray(lse_part, dtype=np.float64)
    n, rows = l.shape
    out = np.empty((rows, D), dtype=np.float64)
    lse = np.empty((rows,), dtype=np.float64)
    _load().oracle_combine(n, rows, _ptr(o), _ptr(l), _ptr(out), _ptr(lse))
    return out, lse


def _row_positions(x: np.ndarray, pos) -> np.ndarray:
    """One int32 position per 512-wide row of x: pos broadcast over x's
    leading axes (e.g. [b, s] positions for [b, s, h, 512] outputs)."""
    lead = x.shape[:-1]
    p = np.asarray(pos, dtype=np.int64)
    p = p.reshape(p.shape + (1,) * (len(lead) - p.ndim))
    return np.ascontiguousarray(np.broadcast_to(p, lead).astype(np.int32)).reshape(-1)


def rope_rotate(x: np.ndarray, pos, theta: float, sign: int = -1) -> np.ndarray:
    """Rotary rotation of dims 448..511 of float64 rows [..., 512]: sign -1
    is the output side's conjugate rotation, +1 the forward one."""
    v = np.ascontiguousarray(x, dtype=np.float64).copy()
    rows = v.size // D
    p = _row_positions(v, pos)
    _load().oracle_rope_rotate(_ptr(v), rows, _ptr(p), float(theta), int(sign))
    return v


def rope_fp8_epilogue(o: np.ndarray, pos, theta: float) -> np.ndarray:
    """The fused epilogue: conjugate rotation of float64 outputs [..., 512]
    and the cast to 528-byte FP8 records [..., 528]."""
    v = np.ascontiguousarray(o, dtype=np.float64)
    rows = v.size // D
    p = _row_positions(v, pos)
    recs = np.empty(v.shape[:-1] + (FP8_RECORD_BYTES,), dtype=np.uint8)
    _load().oracle_rope_fp8_epilogue(_ptr(v), rows, _ptr(p), float(theta), _ptr(recs))
    return recs


def num_threads() -> int:
    return int(_load().oracle_num_threads())
