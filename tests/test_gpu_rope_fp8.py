"""GPU parity of the fused output epilogue (mla_sparse_decode_rope_fp8):
attention output, conjugate rotary embedding of dims 448..511, cast to
528-byte FP8 records, checked against the fp64 oracle (its unrounded
attention output, its rotation and its FP8 encoder).

The GPU's fp32 attention output is within the decode tolerance
(1e-2 + 1e-2 |ref|) of the oracle's; the rotation mixes each pair, so on
dims 448..511 the bound is the sum over the pair; the cast then moves a value
by at most half an E4M3 step under its block scale.  So each decoded GPU
value must lie within that composed bound of the oracle's rotated fp64
value; block scales may differ by one binade (a block maximum near a power
of two).  Most bytes equal the oracle's own encoding: the output carries a
relative error of a few 1e-3 (P is rounded to bf16 for the PV product)
against E4M3 steps of 6-12 %, so a few percent of the values round to the
neighbouring code; at least 90 % must agree.""" 
import numpy as np
import pytest
import torch

import oracle
import synth
from _harness import DeviceWorkload, LSE_ATOL, all_queries, oracle_on, sample_queries

pytestmark = pytest.mark.gpu

THETA = 10000.0


def _step(v, sbyte):
    """One E4M3 step at value v under block scale 2^(sbyte - 127)."""
    sc = np.ldexp(1.0, sbyte.astype(np.int64) - 127)
    x = np.abs(v) / sc
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -9)))
    return np.maximum(2.0 ** (e - 3), 2.0 ** -9) * sc


def _check_records(got, want, ref_rot, ref_out):
    """got / want: uint8 [rows, 528] (GPU, oracle encoding); ref_rot: the
    oracle's rotated fp64 rows; ref_out: its rows before the rotation."""
    got = got.reshape(-1, 528)
    want = want.reshape(-1, 528)
    sg = np.repeat(got[:, 512:].astype(np.int64), 32, axis=1)
    sw = np.repeat(want[:, 512:].astype(np.int64), 32, axis=1)
    assert np.abs(sg - sw).max() <= 1, "block scales differ by more than one binade"
    vg = oracle.dequant_fp8(got).reshape(-1, 512)
    tol = 1e-2 + 1e-2 * np.abs(ref_out)
    pair = np.abs(ref_out[:, 448::2]) + np.abs(ref_out[:, 449::2])
    tol[:, 448::2] = 2e-2 + 1e-2 * pair
    tol[:, 449::2] = 2e-2 + 1e-2 * pair
    bound = tol + 0.5 * _step(vg, sg)
    bad = np.abs(vg - ref_rot) > bound
    assert not bad.any(), f"{bad.sum()} values outside the composed bound"
    same = np.mean(got == want)
    assert same >= 0.90, f"only {same:.4f} of the bytes agree with the oracle's encoding"


def _run(w, queries, positions, num_sms=0):
    dw = DeviceWorkload(w)
    dec = dw.decoder(num_sms)
    dec.error.zero_()
    pos = torch.from_numpy(positions.astype(np.int32)).to(dw.dev)
    out, lse = dec.rope_fp8(dw.q, dw.kv, dw.idx, pos, THETA, dw.xkv, dw.xidx)
    torch.cuda.synchronize()
    assert int(dec.error.item()) == 0
    ref = oracle_on(w, queries)
    qpos = np.array([positions[b, s] for b, s in queries])
    want = oracle.rope_fp8_epilogue(ref["out_f64"], qpos, THETA)      # [n, 1, h, 528]
    rot = oracle.rope_rotate(ref["out_f64"], qpos, THETA, -1)
    got = out.cpu().numpy()
    l = lse.cpu().numpy()
    for j, (b, s) in enumerate(queries):
        _check_records(got[b, s], want[j, 0], rot[j, 0], ref["out_f64"][j, 0])
        gl, wl = l[b, s].astype(np.float64), ref["lse"][j, 0]
        both = np.isneginf(gl) & np.isneginf(wl)
        assert np.all(both | (np.abs(gl - wl) <= LSE_ATOL))
    return out, lse


@pytest.mark.parametrize("cid,batch", [(0, 1), (1, 4), (2, 2), (3, 3)])
def test_rope_fp8_matches_the_oracle(cid, batch):
    """16, 64 and 128 heads, the FP4 extra cache, two query tokens per
    sequence; random positions up to 2^17."""
    w = synth.make_workload(cid, batch=batch, workers=1)
    rng = np.random.default_rng(cid)
    positions = rng.integers(0, 1 << 17, size=(w.cfg.batch, w.cfg.seq_len_q))
    _run(w, all_queries(w), positions)


@pytest.mark.parametrize("cid", [1, 2])
@pytest.mark.parametrize("num_sms", [1, 20, 100000])
def test_rope_fp8_with_any_split_count(cid, num_sms):
    """One part, parts that end one token's split and start the next's,
    one tile per part: every query token's splits are merged before the
    rotation and the cast.  At 128 heads a query token of one split is
    written by the decode kernel itself (every token with one part, none
    with one tile per part)."""
    w = synth.make_workload(cid, batch=3, workers=1)
    positions = (np.array([5, 4096, 131071])[:, None] + 977 * np.arange(w.cfg.seq_len_q)[None, :]) % (1 << 17)
    _run(w, all_queries(w), positions, num_sms=num_sms)


def test_rope_fp8_merge_over_parts():
    """128 heads, fewer parts than query tokens: one-split tokens written by
    the decode kernel, the split ones by the merge over parts."""
    w = synth.make_workload(2, batch=8, workers=1)
    rng = np.random.default_rng(8)
    positions = rng.integers(0, 1 << 17, size=(w.cfg.batch, w.cfg.seq_len_q))
    _run(w, all_queries(w), positions, num_sms=12)


def test_rope_fp8_unaligned_records_match_aligned():
    """Records written to a 4-byte (not 16-byte) aligned buffer -- word
    stores in the 128-head kernel's own epilogue, the merge unchanged -- are
    byte-identical to the aligned run, for one part (every token written by
    the decode kernel) and for the default split."""
    w = synth.make_workload(2, batch=2, workers=1)
    dw = DeviceWorkload(w)
    rng = np.random.default_rng(5)
    pos = torch.from_numpy(rng.integers(0, 1 << 17, size=(w.cfg.batch, w.cfg.seq_len_q)).astype(np.int32)).to(dw.dev)
    shape = (w.cfg.batch, w.cfg.seq_len_q, w.cfg.h_q, 528)
    n = int(np.prod(shape))
    for num_sms in (1, 0):
        dec = dw.decoder(num_sms)
        dec.error.zero_()
        ref, ref_lse = dec.rope_fp8(dw.q, dw.kv, dw.idx, pos, THETA)
        raw = torch.zeros((n + 16,), dtype=torch.uint8, device=dw.dev)
        off = raw[4:4 + n].view(shape)
        assert off.data_ptr() % 16 == 4
        out, lse = dec.rope_fp8(dw.q, dw.kv, dw.idx, pos, THETA, out=off)
        torch.cuda.synchronize()
        assert int(dec.error.item()) == 0
        assert torch.equal(out.cpu(), ref.cpu())
        assert torch.equal(lse.cpu(), ref_lse.cpu())
        assert int(raw[:4].sum()) == 0 and int(raw[4 + n:].sum()) == 0  # nothing written outside


@pytest.mark.parametrize("cid", [1, 2])
def test_rope_fp8_position_zero_and_empty_rows(cid):
    """Position 0 turns nothing (the records are the plain FP8 cast of the
    output); a query token with no valid index gives all-zero codes under
    scale byte 127 and -inf (64 heads through the merge, 128 heads from
    the decode kernel's own epilogue with one part)."""
    w = synth.make_workload(cid, batch=2, workers=1)
    w.idx[1] = -1
    positions = np.zeros((2, w.cfg.seq_len_q), dtype=np.int64)
    out, lse = _run(w, all_queries(w), positions, num_sms=1)
    rec = out[1].cpu().numpy().reshape(-1, 528)
    assert np.all(rec[:, :512] == 0) and np.all(rec[:, 512:] == 127)
    assert torch.isneginf(lse[1]).all()


def test_rope_fp8_full_size_headline_sampled():
    """The 128-head, two-token workload at full size in the benchmark's
    launch configuration, sampled query tokens."""
    w = synth.make_workload(2)
    rng = np.random.default_rng(2)
    positions = rng.integers(0, 1 << 17, size=(w.cfg.batch, w.cfg.seq_len_q))
    _run(w, sample_queries(w, n=3, seed=2), positions)
