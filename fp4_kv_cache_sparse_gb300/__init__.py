"""Python binding of the sm_103a token-sparse MLA decode library (libmla.so).

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels, declared in ``include/mla.h``.  PyTorch supplies device memory
and the current stream.  There is no CPU path: if the library is missing or
a tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import build as _build

__all__ = [
    "MLAError", "Problem", "load", "get_metadata", "sparse_decode", "sparse_decode_rope_fp8", "combine",
    "dequantize", "kv_write",
    "SparseMLADecoder", "decode", "KV_NONE", "KV_FP8_528", "KV_FP4_288", "KV_BF16",
    "DEVERR_BAD_INDEX", "DEVERR_TIMEOUT", "DEVERR_BAD_METADATA", "SCHED_INTS",
]

KV_NONE, KV_FP8_528, KV_FP4_288, KV_BF16 = 0, 1, 2, 3
DEVERR_BAD_INDEX, DEVERR_TIMEOUT, DEVERR_BAD_METADATA = 1, 2, 4
SCHED_INTS = 8
HEAD_DIM = 512
PAGE_SIZE = 64
FP8_RECORD_BYTES = 528
FP4_RECORD_BYTES = 288

STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_WORKSPACE",
          4: "MLA_ERR_CUDA", 5: "MLA_ERR_TIMEOUT"}


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class Problem(ctypes.Structure):
    """mla_problem_t (include/mla.h)."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("seq_len_q", ctypes.c_int32), ("h_q", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("extra_topk", ctypes.c_int32), ("num_pages", ctypes.c_int64), ("extra_num_pages", ctypes.c_int64),
        ("page_size", ctypes.c_int32), ("kv_format", ctypes.c_int32), ("extra_kv_format", ctypes.c_int32),
        ("sm_scale", ctypes.c_float),
    ]

    @classmethod
    def make(cls, batch, seq_len_q, h_q, topk, num_pages, extra_topk=0, extra_num_pages=0,
             sm_scale=None, kv_format=KV_FP8_528, extra_kv_format=None, head_dim=HEAD_DIM,
             page_size=PAGE_SIZE, num_kv_heads=1) -> "Problem":
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(head_dim)
        if extra_kv_format is None:
            extra_kv_format = KV_FP4_288 if extra_topk else KV_NONE
        return cls(batch, seq_len_q, h_q, head_dim, num_kv_heads, topk, extra_topk, num_pages,
                   extra_num_pages, page_size, kv_format, extra_kv_format, sm_scale)


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmla.so (built in-tree by ``build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libmla.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    PP = ctypes.POINTER(Problem)
    lib.mla_get_metadata.argtypes = [PP, I32, P, P, ctypes.POINTER(I32), ctypes.POINTER(SZ), P]
    lib.mla_sparse_decode.argtypes = [PP, P, P, P, P, P, P, P, I32, P, SZ, P, P, P, P]
    lib.mla_sparse_decode_rope_fp8.argtypes = [PP, P, P, P, P, P, P, P, I32, P, SZ, P, ctypes.c_float, P, P, P, P]
    lib.mla_combine.argtypes = [PP, P, P, P, P, P, P]
    lib.mla_dequantize.argtypes = [I32, P, I64, P, P]
    lib.mla_kv_write.argtypes = [I32, P, P, I64, P, I64, P, P]
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_status_string.restype = ctypes.c_char_p
    for f in (lib.mla_get_metadata, lib.mla_sparse_decode, lib.mla_sparse_decode_rope_fp8, lib.mla_combine,
              lib.mla_dequantize, lib.mla_kv_write):
        f.restype = ctypes.c_int
    if path == _build.LIB:
        _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        raise MLAError(status, what)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device (no CPU path)")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def get_metadata(problem: Problem, num_sms: int = 0, device=None, stream=None):
    """Return (sched int32[num_parts, 8], num_splits int32[b*s+1], num_parts, workspace_bytes)."""
    lib = load()
    parts = ctypes.c_int32(0)
    ws = ctypes.c_size_t(0)
    _check(lib.mla_get_metadata(ctypes.byref(problem), num_sms, None, None, ctypes.byref(parts),
                                ctypes.byref(ws), None), "mla_get_metadata (query)")
    device = device or torch.device("cuda", torch.cuda.current_device())
    sched = torch.empty((parts.value, SCHED_INTS), dtype=torch.int32, device=device)
    nsplit = torch.empty((problem.batch * problem.seq_len_q + 1,), dtype=torch.int32, device=device)
    _check(lib.mla_get_metadata(ctypes.byref(problem), num_sms, _ptr(sched), _ptr(nsplit),
                                ctypes.byref(parts), ctypes.byref(ws), _stream(stream)), "mla_get_metadata")
    return sched, nsplit, parts.value, ws.value


def sparse_decode(problem: Problem, q, kv, indices, sched, num_splits, num_parts, workspace,
                  out, lse, extra_kv=None, extra_indices=None, error=None, stream=None):
    lib = load()
    _check(lib.mla_sparse_decode(ctypes.byref(problem), _ptr(q), _ptr(kv), _ptr(indices), _ptr(extra_kv),
                                 _ptr(extra_indices), _ptr(sched), _ptr(num_splits), num_parts,
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _ptr(out), _ptr(lse), _ptr(error), _stream(stream)), "mla_sparse_decode")


def sparse_decode_rope_fp8(problem: Problem, q, kv, indices, sched, num_splits, num_parts, workspace,
                           positions, rope_theta, out_fp8, lse, extra_kv=None, extra_indices=None, error=None,
                           stream=None):
    """The decode step with the fused output epilogue: conjugate rotary
    embedding of dims 448..511 and the cast to 528-byte FP8 records
    (out_fp8 uint8 [b, s, h, 528]); positions int32 [b, s]."""
    lib = load()
    _check(lib.mla_sparse_decode_rope_fp8(ctypes.byref(problem), _ptr(q), _ptr(kv), _ptr(indices), _ptr(extra_kv),
                                          _ptr(extra_indices), _ptr(sched), _ptr(num_splits), num_parts,
                                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _ptr(positions), float(rope_theta), _ptr(out_fp8), _ptr(lse),
                                          _ptr(error), _stream(stream)), "mla_sparse_decode_rope_fp8")


def combine(problem: Problem, num_splits, o_partial, lse_partial, out, lse, stream=None):
    lib = load()
    _check(lib.mla_combine(ctypes.byref(problem), _ptr(num_splits), _ptr(o_partial), _ptr(lse_partial),
                           _ptr(out), _ptr(lse), _stream(stream)), "mla_combine")


def kv_write(latents: torch.Tensor, slots: torch.Tensor, pool: torch.Tensor, kv_format: int = KV_FP8_528,
             num_pages: int = None, error: torch.Tensor = None, stream=None) -> None:
    """Quantize bf16 latents [n, 512] into FP8 (528-byte) or FP4 (288-byte)
    records and store each at its slot (page*64 + offset, -1 = skip) of the
    uint8 pool [num_pages, 64, record] (or [tokens, record])."""
    lib = load()
    rec = FP8_RECORD_BYTES if kv_format == KV_FP8_528 else FP4_RECORD_BYTES
    if num_pages is None:
        num_pages = pool.numel() // (PAGE_SIZE * rec)
    n = latents.shape[0] if latents.dim() > 0 else 0
    _check(lib.mla_kv_write(kv_format, _ptr(latents), _ptr(slots), n, _ptr(pool), num_pages, _ptr(error),
                            _stream(stream)), "mla_kv_write")


def dequantize(records: torch.Tensor, kv_format: int = KV_FP8_528, stream=None) -> torch.Tensor:
    """uint8 [n, 528|288] records -> bf16 [n, 512], with the decode kernel's dequantization."""
    lib = load()
    n = records.shape[0]
    out = torch.empty((n, HEAD_DIM), dtype=torch.bfloat16, device=records.device)
    _check(lib.mla_dequantize(kv_format, _ptr(records), n, _ptr(out), _stream(stream)), "mla_dequantize")
    return out


class SparseMLADecoder:
    """Metadata and workspace planned once for a problem shape; one call per step."""

    def __init__(self, problem: Problem, device=None, num_sms: int = 0, stream=None):
        self.problem = problem
        self.device = device or torch.device("cuda", torch.cuda.current_device())
        self.sched, self.num_splits, self.num_parts, self.ws_bytes = get_metadata(
            problem, num_sms, self.device, stream)
        self.workspace = torch.empty((max(self.ws_bytes, 16),), dtype=torch.uint8, device=self.device)
        self.error = torch.zeros((1,), dtype=torch.int32, device=self.device)

    def __call__(self, q, kv, indices, extra_kv=None, extra_indices=None, out=None, lse=None, stream=None):
        p = self.problem
        if out is None:
            out = torch.empty((p.batch, p.seq_len_q, p.h_q, HEAD_DIM), dtype=torch.bfloat16, device=q.device)
        if lse is None:
            lse = torch.empty((p.batch, p.seq_len_q, p.h_q), dtype=torch.float32, device=q.device)
        sparse_decode(p, q, kv, indices, self.sched, self.num_splits, self.num_parts, self.workspace,
                      out, lse, extra_kv, extra_indices, self.error, stream)
        return out, lse

    def rope_fp8(self, q, kv, indices, positions, rope_theta=10000.0, extra_kv=None, extra_indices=None,
                 out=None, lse=None, stream=None):
        """Decode with the fused epilogue; returns (FP8 records uint8 [b, s, h, 528], lse)."""
        p = self.problem
        if out is None:
            out = torch.empty((p.batch, p.seq_len_q, p.h_q, FP8_RECORD_BYTES), dtype=torch.uint8, device=q.device)
        if lse is None:
            lse = torch.empty((p.batch, p.seq_len_q, p.h_q), dtype=torch.float32, device=q.device)
        sparse_decode_rope_fp8(p, q, kv, indices, self.sched, self.num_splits, self.num_parts, self.workspace,
                               positions, rope_theta, out, lse, extra_kv, extra_indices, self.error, stream)
        return out, lse


def decode(q, kv, indices, extra_kv=None, extra_indices=None, sm_scale=None):
    """One-shot decode.  q bf16 [b, s, h, 512]; kv uint8 [pages, 64, 528] (or
    [tokens, 528]); indices int32 [b, s, topk]; optional FP4 extra cache.
    Returns (out bf16 [b, s, h, 512], lse float32 [b, s, h])."""
    b, s, h, d = q.shape
    num_pages = kv.numel() // (PAGE_SIZE * FP8_RECORD_BYTES)
    xtopk = extra_indices.shape[-1] if extra_indices is not None else 0
    xpages = extra_kv.numel() // (PAGE_SIZE * FP4_RECORD_BYTES) if extra_kv is not None else 0
    prob = Problem.make(b, s, h, indices.shape[-1], num_pages, extra_topk=xtopk, extra_num_pages=xpages,
                        sm_scale=sm_scale, head_dim=d)
    return SparseMLADecoder(prob, q.device)(q, kv, indices, extra_kv, extra_indices)
