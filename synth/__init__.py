"""Seeded synthetic inputs for token-sparse MLA decode.

This module serves both the oracle and the GPU path and holds none of the
decode arithmetic: it draws queries, latents and index sets and *encodes*
latents into the cache record formats (the inverse direction of what the
decode path computes).  Decoding, attention and merging live in ``oracle/``
and in the CUDA library, separately.

Workloads (all values N(0, 1), fixed seeds 1000 + workload id, numpy PCG64):

  0 tiny_fp8         b=1,   s=1, h=16,  pool 128 tokens, topk 64 distinct,
                     6 entries (10 %) set to -1 at random slots.
  1 fp8_b64_h64      b=64,  s=1, h=64,  pool 32768 tokens per sequence,
                     topk 2048 distinct uniform, last 20 slots (1 %) -1.
  2 fp8_b128_s2_h128 b=128, s=2, h=128, pool 131072 tokens per sequence,
                     topk 2048 = 1024 distinct from the last 4096 positions +
                     1024 distinct from the rest, shuffled, last 20 slots -1;
                     the two query tokens draw independently.
  3 fp8_fp4_b64_h64  b=64,  s=1, h=64,  FP8 pool 65536 / FP4 extra pool 16384
                     tokens per sequence, topk 2048 + extra topk 512, no -1.
  4 long_dense_b32_h16  b=32, s=1, h=16, pool 1048576 tokens per sequence,
                     the last 65536 positions, contiguous, no -1.
  5 long_sparse_b32_h16 same pool, 8192 distinct uniform positions, no -1.

Sequence b owns the contiguous pages [b*P/64, (b+1)*P/64) of its pool, so an
index is b*P + position = page_block*64 + offset.  Only referenced records
are generated; the rest of a pool is filled with POISON_BYTE, which decodes
to huge or infinite values, so a read of an unselected record shows up in the
output.
"""
from __future__ import annotations

import dataclasses
import math
import os
import sys
from typing import Optional

import numpy as np

D = 512
FP8_RECORD_BYTES = 528
FP4_RECORD_BYTES = 288
PAGE_SIZE = 64
POISON_BYTE = 0xFE
SEED_BASE = 1000


@dataclasses.dataclass(frozen=True)
class Config:
    id: int
    name: str
    batch: int
    seq_len_q: int
    h_q: int
    pool: int                 # tokens per sequence, main FP8 cache
    topk: int
    neg: int = 0              # number of -1 entries per query
    neg_mode: str = "trailing"  # "trailing" | "random"
    recent_window: int = 0    # >0: half the picks from the last recent_window positions
    contiguous: bool = False  # pick the last topk positions in order
    extra_pool: int = 0       # tokens per sequence, FP4 extra cache
    extra_topk: int = 0

    @property
    def sm_scale(self) -> np.float32:
        return np.float32(1.0 / math.sqrt(D))


CONFIGS = [
    Config(0, "tiny_fp8", 1, 1, 16, 128, 64, neg=6, neg_mode="random"),
    Config(1, "fp8_b64_h64", 64, 1, 64, 32768, 2048, neg=20),
    Config(2, "fp8_b128_s2_h128", 128, 2, 128, 131072, 2048, neg=20, recent_window=4096),
    Config(3, "fp8_fp4_b64_h64", 64, 1, 64, 65536, 2048, extra_pool=16384, extra_topk=512),
    Config(4, "long_dense_b32_h16", 32, 1, 16, 1048576, 65536, contiguous=True),
    Config(5, "long_sparse_b32_h16", 32, 1, 16, 1048576, 8192),
    # Prefill-shaped: one sequence, 1024 query tokens each with its own 2048
    # indices (the same index semantics at seq_len_q >> 1).
    Config(6, "prefill_b1_s1024_h128", 1, 1024, 128, 65536, 2048, neg=20, recent_window=4096),
]
BY_NAME = {c.name: c for c in CONFIGS}


@dataclasses.dataclass
class Workload:
    cfg: Config
    q_bits: np.ndarray            # uint16 [b, s, h, 512], bf16 patterns
    idx: np.ndarray               # int32 [b, s, topk]
    pool_tokens: int              # total main-pool tokens (all sequences)
    ref_pos: np.ndarray           # int64 [n], sorted unique referenced positions
    ref_rec: np.ndarray           # uint8 [n, 528]
    extra_idx: Optional[np.ndarray] = None
    extra_pool_tokens: int = 0
    extra_ref_pos: Optional[np.ndarray] = None
    extra_ref_rec: Optional[np.ndarray] = None

    @property
    def sm_scale(self) -> np.float32:
        return self.cfg.sm_scale


# ---------------------------------------------------------------------------
# Encoders (test-input production only).
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 bit patterns, round to nearest even (finite input)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def _pow2(e: np.ndarray) -> np.ndarray:
    """2.0 ** e for integer e in the normal binary64 range, built from bits."""
    return ((np.asarray(e, dtype=np.int64) + 1023) << 52).view(np.float64)


def _e4m3_encode(v: np.ndarray):
    """Round float64 values to E4M3FN (ties to even, saturating at +-448).

    Returns (codes uint8, rounded values float64)."""
    neg = np.signbit(v)
    a = np.minimum(np.abs(v), 448.0)
    sub = a < 2.0 ** -6
    E = ((a.view(np.uint64) >> 52).astype(np.int64) - 1023)
    E = np.where(sub, -6, E)                 # exponent of the quantum's binade
    n = np.rint(a * _pow2(3 - E))            # a / 2^(E-3), exact scaling
    carry = (~sub) & (n >= 16)
    E = E + carry
    n = np.where(carry, 8.0, n)
    ni = n.astype(np.int64)
    code = np.where(sub, ni, ((E + 7) << 3) | (ni - 8))
    code = code | np.where(neg, 0x80, 0)
    val = n * _pow2(E - 3)
    val = np.where(neg, -val, val)
    return code.astype(np.uint8), val


_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_E2M1_MID = (_E2M1_GRID[1:] + _E2M1_GRID[:-1]) / 2.0


def _e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Round float64 values to e2m1 codes (ties to even code, saturating at 6)."""
    neg = np.signbit(v)
    a = np.minimum(np.abs(v), 6.0)
    i = np.searchsorted(_E2M1_MID, a, side="left")
    tie = (i < len(_E2M1_MID)) & (a == _E2M1_MID[np.minimum(i, len(_E2M1_MID) - 1)])
    i = np.where(tie & (i % 2 == 1), i + 1, i)
    return (i | np.where(neg, 8, 0)).astype(np.uint8)


def encode_fp8_records(x: np.ndarray) -> np.ndarray:
    """Latents float32 [n, 512] -> 528-byte records.

    Per 32-value block: scale exponent e = ceil(log2(amax / 448)) (exact, via
    frexp), e8m0 byte 127 + e, values x * 2^-e rounded to E4M3FN.  An all-zero
    block gets byte 127."""
    n = x.shape[0]
    xb = x.astype(np.float64).reshape(n, 16, 32)
    amax = np.abs(xb).max(axis=2)
    f, ex = np.frexp(amax / 448.0)
    e = np.where(f == 0.5, ex - 1, ex)
    e = np.where(amax == 0, 0, e)
    e = np.clip(e, -127, 127)
    codes, _ = _e4m3_encode(xb * np.ldexp(1.0, -e)[..., None])
    rec = np.empty((n, FP8_RECORD_BYTES), dtype=np.uint8)
    rec[:, :512] = codes.reshape(n, 512)
    rec[:, 512:] = (127 + e).astype(np.uint8)
    return rec


def encode_fp4_records(x: np.ndarray) -> np.ndarray:
    """Latents float32 [n, 512] -> 288-byte records.

    Per 16-value block: scale s = amax / 6 rounded to E4M3FN, values x / s
    rounded to e2m1 (all zero when s rounds to 0).  Byte k packs value 2k in
    the low nibble and value 2k+1 in the high nibble."""
    n = x.shape[0]
    xb = x.astype(np.float64).reshape(n, 32, 16)
    amax = np.abs(xb).max(axis=2)
    scode, sval = _e4m3_encode(amax / 6.0)
    safe = np.where(sval == 0, 1.0, sval)
    codes = _e2m1_encode(xb / safe[..., None])
    codes = np.where((sval == 0)[..., None], 0, codes).astype(np.uint8).reshape(n, 512)
    rec = np.empty((n, FP4_RECORD_BYTES), dtype=np.uint8)
    rec[:, :256] = codes[:, 0::2] | (codes[:, 1::2] << 4)
    rec[:, 256:] = scode
    return rec


# ---------------------------------------------------------------------------
# Index sets.
# ---------------------------------------------------------------------------

def _positions(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    """Per-sequence positions of one query token, int64 [topk] (before -1)."""
    P = cfg.pool
    if cfg.contiguous:
        return np.arange(P - cfg.topk, P, dtype=np.int64)
    if cfg.recent_window:
        half = cfg.topk // 2
        recent = P - cfg.recent_window + rng.choice(cfg.recent_window, half, replace=False)
        rest = rng.choice(P - cfg.recent_window, cfg.topk - half, replace=False)
        pos = np.concatenate([recent, rest]).astype(np.int64)
        rng.shuffle(pos)
        return pos
    return rng.choice(P, cfg.topk, replace=False).astype(np.int64)


def _apply_neg(cfg: Config, ids: np.ndarray, rng: np.random.Generator) -> None:
    if cfg.neg == 0:
        return
    if cfg.neg_mode == "random":
        slots = rng.choice(ids.shape[-1], cfg.neg, replace=False)
        ids[slots] = -1
    else:
        ids[-cfg.neg:] = -1


CHUNK = 2048


def _encode_chunk(args):
    base_seed, kind, c, n = args
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([base_seed, kind, c])))
    lat = rng.standard_normal((n, D), dtype=np.float32)
    return encode_fp8_records(lat) if kind == 1 else encode_fp4_records(lat)


def _encode_chunks(base_seed: int, kind: int, n: int, workers: Optional[int]) -> np.ndarray:
    """Latents of n records, drawn chunk by chunk from seeds (base, kind, chunk),
    so that the bytes do not depend on how many processes encode them."""
    R = FP8_RECORD_BYTES if kind == 1 else FP4_RECORD_BYTES
    out = np.empty((n, R), dtype=np.uint8)
    jobs = [(base_seed, kind, c, min(CHUNK, n - c * CHUNK)) for c in range((n + CHUNK - 1) // CHUNK)]
    if workers is None:
        workers = min(os.cpu_count() or 1, 32) if len(jobs) > 32 else 1
        main = sys.modules.get("__main__")
        if not os.path.exists(getattr(main, "__file__", "") or ""):
            workers = 1       # spawn needs an importable main module
    if workers > 1:
        import concurrent.futures
        import multiprocessing
        ctx = multiprocessing.get_context("spawn")
        with concurrent.futures.ProcessPoolExecutor(workers, mp_context=ctx) as ex:
            for (_, _, c, m), rec in zip(jobs, ex.map(_encode_chunk, jobs, chunksize=4)):
                out[c * CHUNK:c * CHUNK + m] = rec
    else:
        for (_, _, c, m) in jobs:
            out[c * CHUNK:c * CHUNK + m] = _encode_chunk((base_seed, kind, c, m))
    return out


def make_workload(cfg: Config | int | str, seed: Optional[int] = None,
                  scattered_neg: bool = False, batch: Optional[int] = None,
                  workers: Optional[int] = None, pool: Optional[int] = None) -> Workload:
    """Draw the workload of a configuration.

    scattered_neg moves the -1 entries of a 'trailing' configuration to random
    slots.  batch / pool override the number of sequences and the tokens per
    sequence: a smaller workload of the same family (its values are not a
    subset of the full draw)."""
    if isinstance(cfg, int):
        cfg = CONFIGS[cfg]
    elif isinstance(cfg, str):
        cfg = BY_NAME[cfg]
    if batch is not None and batch != cfg.batch:
        cfg = dataclasses.replace(cfg, batch=batch)
    if pool is not None and pool != cfg.pool:
        assert pool % PAGE_SIZE == 0 and pool >= cfg.topk and pool > cfg.recent_window
        cfg = dataclasses.replace(cfg, pool=pool)
    if scattered_neg:
        cfg = dataclasses.replace(cfg, neg_mode="random")
    base_seed = SEED_BASE + cfg.id if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([base_seed, 0])))
    b, s, h = cfg.batch, cfg.seq_len_q, cfg.h_q

    q = rng.standard_normal((b, s, h, D), dtype=np.float32)
    q_bits = f32_to_bf16_bits(q)
    del q

    idx = np.empty((b, s, cfg.topk), dtype=np.int32)
    xidx = np.empty((b, s, cfg.extra_topk), dtype=np.int32) if cfg.extra_topk else None
    for bi in range(b):
        for si in range(s):
            pos = _positions(cfg, rng)
            ids = (bi * cfg.pool + pos).astype(np.int64)
            _apply_neg(cfg, ids, rng)
            idx[bi, si] = ids
            if xidx is not None:
                xpos = rng.choice(cfg.extra_pool, cfg.extra_topk, replace=False).astype(np.int64)
                xidx[bi, si] = bi * cfg.extra_pool + xpos

    def records(ids: np.ndarray, kind: int):
        pos = np.unique(ids[ids >= 0].astype(np.int64))
        return pos, _encode_chunks(base_seed, kind, pos.shape[0], workers)

    ref_pos, ref_rec = records(idx, 1)
    w = Workload(cfg=cfg, q_bits=q_bits, idx=idx, pool_tokens=b * cfg.pool,
                 ref_pos=ref_pos, ref_rec=ref_rec)
    if xidx is not None:
        w.extra_idx = xidx
        w.extra_pool_tokens = b * cfg.extra_pool
        w.extra_ref_pos, w.extra_ref_rec = records(xidx, 2)
    return w


# ---------------------------------------------------------------------------
# Pool views.
# ---------------------------------------------------------------------------

def full_pool(w: Workload, extra: bool = False) -> np.ndarray:
    """Host copy of a whole pool (poison where unreferenced); small pools only."""
    if extra:
        n, R, pos, rec = w.extra_pool_tokens, FP4_RECORD_BYTES, w.extra_ref_pos, w.extra_ref_rec
    else:
        n, R, pos, rec = w.pool_tokens, FP8_RECORD_BYTES, w.ref_pos, w.ref_rec
    pool = np.full((n, R), POISON_BYTE, dtype=np.uint8)
    pool[pos] = rec
    return pool


def compact(w: Workload, queries) -> dict:
    """Inputs of a subset of query tokens with their pools compacted.

    queries: list of (b, s).  The referenced records are gathered into a small
    pool and the indices renumbered to it (-1 stays -1), so that a CPU
    reference can run on a handful of queries of a multi-GB workload; the
    record bytes a query sees are unchanged."""
    qs = list(queries)
    q = np.stack([w.q_bits[bi, si] for bi, si in qs])[:, None]       # [n,1,h,512]
    ids = np.stack([w.idx[bi, si] for bi, si in qs])[:, None]         # [n,1,topk]
    out = dict(q_bits=q)

    def remap(ids, pos, rec):
        # Entries that name no generated record (outside the contract) become
        # -2, which a reference skips just as it skips out-of-range entries.
        loc = np.searchsorted(pos, np.where(ids >= 0, ids, 0))
        loc = np.minimum(loc, max(pos.shape[0] - 1, 0))
        known = (ids >= 0) & (pos.shape[0] > 0) & (pos[loc] == ids)
        uniq, inv = np.unique(loc[known], return_inverse=True)
        new = np.where(ids == -1, -1, -2).astype(np.int32)
        new[known] = inv.astype(np.int32)
        return new, rec[uniq]

    out["idx"], out["kv"] = remap(ids, w.ref_pos, w.ref_rec)
    if w.extra_idx is not None:
        xids = np.stack([w.extra_idx[bi, si] for bi, si in qs])[:, None]
        out["extra_idx"], out["extra_kv"] = remap(xids, w.extra_ref_pos, w.extra_ref_rec)
    return out


def flops(w: Workload) -> float:
    """Algorithmic FLOPs: 4 * 512 per (head, valid selected token)."""
    t = int((w.idx >= 0).sum())
    if w.extra_idx is not None:
        t += int((w.extra_idx >= 0).sum())
    return 4.0 * D * w.cfg.h_q * t


def kv_bytes(w: Workload) -> float:
    """Algorithmic KV bytes: each valid selected record once per query token."""
    t = int((w.idx >= 0).sum()) * FP8_RECORD_BYTES
    if w.extra_idx is not None:
        t += int((w.extra_idx >= 0).sum()) * FP4_RECORD_BYTES
    return float(t)
