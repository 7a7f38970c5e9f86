"""GPU decode parity against the fp64 oracle, element by element.

Tolerances: |out - ref| <= 1e-2 + 1e-2 |ref| (bf16 outputs), |lse - ref| <=
1e-3 (natural log).  Every pool is filled with a poison byte wherever no
index points, so a read of an unselected record would show in the output.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import fp4_kv_cache_sparse_gb300 as mla
import oracle
import synth
from _harness import DeviceWorkload, all_queries, compare, sample_queries

pytestmark = pytest.mark.gpu

REDUCED_BATCH = {0: 1, 1: 4, 2: 2, 3: 4, 4: 1, 5: 3}


@pytest.mark.parametrize("cid", [0, 1, 2, 3, 4, 5])
def test_reduced_configs_all_queries(cid):
    """Every query token of each workload family at a batch the oracle
    finishes in seconds (several tiles per query, ragged -1 tails)."""
    w = synth.make_workload(cid, batch=REDUCED_BATCH[cid], workers=1)
    dw = DeviceWorkload(w)
    out, lse, err = dw.run()
    assert err == 0
    compare(out, lse, w, all_queries(w))


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5, 6])
def test_full_size_sampled_queries(cid):
    """The full workload in the launch configuration the benchmark times;
    sampled query tokens against the oracle (random ones plus the first two
    that the schedule splits over parts, so that the merge is checked at full
    size), the rest checked for finiteness and the -inf/0 convention."""
    w = synth.make_workload(cid)
    dw = DeviceWorkload(w)
    dec = dw.decoder()
    out, lse, err = dw.run(dec=dec)
    assert err == 0
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    qs = all_queries(w)
    splits = np.diff(dec.num_splits.cpu().numpy())
    split_q = [qs[j] for j in np.nonzero(splits > 1)[0][:2]]
    picked = sorted(set(sample_queries(w, n=3, seed=cid)) | set(split_q))
    compare(out, lse, w, picked)


def test_scattered_skips():
    for cid in (1, 2):
        w = synth.make_workload(cid, batch=2, scattered_neg=True, workers=1)
        out, lse, err = DeviceWorkload(w).run()
        compare(out, lse, w, all_queries(w))


def _custom(h_q, topk, pool, idx, q_scale=1.0, seed=0, xpool=0, xidx=None, s=1):
    """A workload from explicit index arrays (idx int [b, s, topk])."""
    rng = np.random.default_rng(seed)
    b = idx.shape[0]
    cfg = synth.Config(99, "custom", b, s, h_q, pool, topk,
                       extra_pool=xpool, extra_topk=0 if xidx is None else xidx.shape[-1])
    q = (rng.standard_normal((b, s, h_q, 512), dtype=np.float32) * q_scale).astype(np.float32)
    pos = np.unique(idx[(idx >= 0) & (idx < pool * b)])
    rec = synth.encode_fp8_records(rng.standard_normal((pos.shape[0], 512), dtype=np.float32))
    w = synth.Workload(cfg=cfg, q_bits=synth.f32_to_bf16_bits(q), idx=idx.astype(np.int32),
                       pool_tokens=pool * b, ref_pos=pos.astype(np.int64), ref_rec=rec)
    if xidx is not None:
        xpos = np.unique(xidx[xidx >= 0])
        w.extra_idx = xidx.astype(np.int32)
        w.extra_pool_tokens = xpool * b
        w.extra_ref_pos = xpos.astype(np.int64)
        w.extra_ref_rec = synth.encode_fp4_records(rng.standard_normal((xpos.shape[0], 512), dtype=np.float32))
    return w


def _random_idx(rng, b, s, topk, pool, neg=0.0):
    idx = np.stack([np.stack([bi * pool + rng.choice(pool, topk, replace=False) for _ in range(s)])
                    for bi in range(b)])
    if neg:
        idx[rng.random(idx.shape) < neg] = -1
    return idx


@pytest.mark.parametrize("h_q", [16, 32, 128])
@pytest.mark.parametrize("num_sms", [0, 7])
def test_three_query_tokens_per_sequence(h_q, num_sms):
    """seq_len_q = 3 (odd), each query token of a sequence with its own
    indices into the sequence's pool; 7 SMs give parts that cut query tokens
    of different sequences."""
    rng = np.random.default_rng(h_q + num_sms)
    idx = _random_idx(rng, 3, 3, 300, 640, neg=0.02)
    w = _custom(h_q, 300, 640, idx, s=3, seed=h_q)
    out, lse, err = DeviceWorkload(w).run(num_sms=num_sms)
    assert err == 0
    compare(out, lse, w, all_queries(w))


@pytest.mark.parametrize("h_q", [16, 32, 64, 128])
@pytest.mark.parametrize("topk", [1, 127, 129, 300])
def test_heads_and_ragged_topk(h_q, topk):
    rng = np.random.default_rng(h_q * 1000 + topk)
    idx = _random_idx(rng, 3, 1, topk, 512, neg=0.1)
    w = _custom(h_q, topk, 512, idx, seed=topk)
    out, lse, err = DeviceWorkload(w).run()
    assert err == 0
    compare(out, lse, w, all_queries(w))


@pytest.mark.parametrize("h_q", [16, 64, 128])
@pytest.mark.parametrize("num_sms", [0, 12])
def test_all_skipped_rows_give_zero_and_neg_inf(h_q, num_sms):
    """Query tokens with no valid index give +0 and -inf; partly masked
    tiles and sub-tiles around them.  Row 1 is all -1; row 3 has its first
    128-slot tile empty and the second partly valid; row 2 has its first
    64-token half-tile empty and the second half valid; row 0 has the first
    half-tile of its third tile empty.  With 12 SMs every query token is
    split over several parts, so some splits start on an empty half-tile or
    hold no valid token at all."""
    rng = np.random.default_rng(7)
    idx = _random_idx(rng, 4, 1, 400, 512)
    idx[1] = -1
    idx[3, 0, :130] = -1          # first tile empty, second partly valid
    idx[2, 0, :64] = -1           # first half-tile empty, second half valid
    idx[0, 0, 256:320] = -1       # third tile: first half empty
    w = _custom(h_q, 400, 512, idx)
    out, lse, err = DeviceWorkload(w).run(num_sms=num_sms)
    assert err == 0
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    assert not torch.signbit(out[1].float()).any()
    compare(out, lse, w, all_queries(w))


@pytest.mark.parametrize("h_q", [16, 64, 128])
def test_extra_cache_joint_softmax_and_extra_only_rows(h_q):
    """One softmax over the FP8 main cache and the FP4 extra cache; a row
    attended through the extra cache alone.  128 heads with an extra cache
    run as two 64-head groups on the swap-AB kernel."""
    rng = np.random.default_rng(8)
    idx = _random_idx(rng, 3, 1, 256, 512, neg=0.05)
    xidx = _random_idx(rng, 3, 1, 130, 192, neg=0.05)
    idx[2] = -1                    # this row is attended through the extra cache alone
    w = _custom(h_q, 256, 512, idx, xpool=192, xidx=xidx)
    out, lse, err = DeviceWorkload(w).run()
    assert err == 0
    compare(out, lse, w, all_queries(w))


@pytest.mark.parametrize("h_q", [16, 64, 128])
def test_duplicate_indices_count_twice(h_q):
    rng = np.random.default_rng(9)
    idx = _random_idx(rng, 2, 1, 100, 320)
    idx[:, :, 50:] = idx[:, :, :50]
    w = _custom(h_q, 100, 320, idx)
    out, lse, _ = DeviceWorkload(w).run()
    compare(out, lse, w, all_queries(w))


@pytest.mark.parametrize("h_q", [16, 64, 128])
def test_first_and_last_pool_tokens(h_q):
    """Indices naming token 0 and the pool's last token (the last row of the
    128-head kernel's row-gather tensor, the last record the other kernel
    loads), in the first and the last slot of a row whose last tile is
    ragged, from both sequences."""
    rng = np.random.default_rng(17)
    b, topk, pool = 2, 300, 320
    idx = _random_idx(rng, b, 1, topk, pool)
    last = pool * b - 1
    idx[0, 0, 0], idx[0, 0, topk - 1] = 0, last
    idx[b - 1, 0, 0], idx[b - 1, 0, topk - 1] = last, 0
    w = _custom(h_q, topk, pool, idx)
    out, lse, err = DeviceWorkload(w).run()
    assert err == 0
    compare(out, lse, w, all_queries(w))


@pytest.mark.parametrize("h_q", [32, 64, 128])
def test_bad_indices_are_skipped_and_flagged(h_q):
    """Entries past the pool or negative other than -1 are skipped on both
    sides and flagged; one bad entry sits in the first half-tile, one in the
    second half of the second tile."""
    rng = np.random.default_rng(10)
    idx = _random_idx(rng, 2, 1, 150, 448)
    idx[0, 0, 5] = 2 * 448 + 7       # past the pool (7 pages per sequence)
    idx[1, 0, 140] = -5              # negative, not -1
    idx[1, 0, 77] = 1 << 30          # far past the pool
    w = _custom(h_q, 150, 448, idx)
    out, lse, err = DeviceWorkload(w).run()
    assert err & mla.DEVERR_BAD_INDEX
    assert err & ~mla.DEVERR_BAD_INDEX == 0
    compare(out, lse, w, all_queries(w))


def test_large_scores_exercise_rescaling():
    """Scores spread over many units: the running max moves by more than the
    lazy-rescale threshold inside a query token."""
    rng = np.random.default_rng(11)
    idx = _random_idx(rng, 3, 2, 1024, 2048)
    w = _custom(64, 1024, 2048, idx, q_scale=6.0, s=2)
    out, lse, _ = DeviceWorkload(w).run()
    compare(out, lse, w, all_queries(w))


@pytest.mark.parametrize("h_q", [16, 64, 128])
def test_large_block_scales_in_the_decode(h_q):
    """FP8 block scales beyond 2^15 (scale bytes above 142, which the
    dequantization takes in two multiplies) through each decode kernel's own
    scale handling: per-quarter loads (16 heads), per-tile loads (64 heads)
    and the 128-head kernel's staged scales.  Multiplying every latent by
    2^24 leaves the E4M3 codes as they are and raises each scale byte by 24;
    with the queries multiplied by 2^-24 the scores do not change.  So the
    scaled problem must give exactly 2^24 times the outputs and the same LSE
    as the unscaled one, which is checked against the oracle.  Half the
    latents are 2^-16 smaller, so that scaled warps see both dequantization
    paths."""
    rng = np.random.default_rng(31 + h_q)
    b, topk, pool = 2, 1024, 4096
    idx = _random_idx(rng, b, 1, topk, pool, neg=0.01)
    pos = np.unique(idx[idx >= 0])
    data = rng.standard_normal((pos.shape[0], 512), dtype=np.float32)
    data *= np.where(rng.random(pos.shape[0]) < 0.5, 1.0, 2.0 ** -16).astype(np.float32)[:, None]
    rec_small = synth.encode_fp8_records(data)
    rec_big = synth.encode_fp8_records(data * np.float32(2.0 ** 24))
    assert np.array_equal(rec_small[:, :512], rec_big[:, :512])
    assert np.array_equal(rec_small[:, 512:].astype(np.int32) + 24, rec_big[:, 512:].astype(np.int32))
    assert (rec_small[:, 512:] <= 142).all()
    assert (rec_big[:, 512:] > 142).any() and (rec_big[:, 512:] <= 142).any()
    q = rng.standard_normal((b, 1, h_q, 512), dtype=np.float32)
    cfg = synth.Config(99, "custom", b, 1, h_q, pool, topk)

    def run(rec, qs):
        w = synth.Workload(cfg=cfg, q_bits=synth.f32_to_bf16_bits(qs), idx=idx.astype(np.int32),
                           pool_tokens=pool * b, ref_pos=pos.astype(np.int64), ref_rec=rec)
        out, lse, err = DeviceWorkload(w).run()
        assert err == 0
        return w, out, lse

    w, out_s, lse_s = run(rec_small, q)
    _, out_b, lse_b = run(rec_big, q * np.float32(2.0 ** -24))
    compare(out_s, lse_s, w, all_queries(w))
    assert torch.equal(out_b.float(), out_s.float() * 2.0 ** 24)
    assert torch.equal(lse_b, lse_s)


@pytest.mark.parametrize("h_q", [64, 128])
def test_growing_scores_move_the_max_every_tile(h_q):
    """Every query row shares a component along one unit direction u, and the
    keys of 128-slot tile t carry 8t along u: each tile's scores sit about ten
    log2 units above the previous tile's, past the lazy-rescale threshold, so
    the running maximum moves, and O and the row sums are rescaled, on every
    tile.  Values stay of order one, so the bf16 P keeps the usual error."""
    rng = np.random.default_rng(21)
    b, topk, pool = 2, 1024, 4096
    idx = _random_idx(rng, b, 1, topk, pool)
    slot_of = {}
    for bi in range(b):
        for t in range(topk):
            slot_of[int(idx[bi, 0, t])] = t
    pos = np.array(sorted(slot_of), dtype=np.int64)
    u = rng.standard_normal(512).astype(np.float32)
    u /= np.linalg.norm(u)
    lift = np.array([8.0 * (slot_of[int(x)] // 128) for x in pos], dtype=np.float32)
    data = rng.standard_normal((pos.shape[0], 512), dtype=np.float32) + lift[:, None] * u[None, :]
    cfg = synth.Config(99, "custom", b, 1, h_q, pool, topk)
    q = rng.standard_normal((b, 1, h_q, 512), dtype=np.float32) + 20.0 * u
    w = synth.Workload(cfg=cfg, q_bits=synth.f32_to_bf16_bits(q), idx=idx.astype(np.int32),
                       pool_tokens=pool * b, ref_pos=pos, ref_rec=synth.encode_fp8_records(data))
    out, lse, _ = DeviceWorkload(w).run()
    compare(out, lse, w, all_queries(w))


@pytest.mark.parametrize("cid", [1, 2])
@pytest.mark.parametrize("num_sms", [1, 3, 20, 152, 100000])
def test_split_counts_do_not_change_results(num_sms, cid):
    """From one part (no split) to one tile per part (every query split into
    all its tiles); 64 heads and 128 heads, merged by the combine kernel.
    20 SMs give parts of 10 tiles over 16-tile query tokens, so some parts
    end one token's split and start the next's."""
    w = synth.make_workload(cid, batch=3, workers=1)
    dw = DeviceWorkload(w)
    out, lse, err = dw.run(num_sms=num_sms)
    assert err == 0
    compare(out, lse, w, all_queries(w))


@pytest.mark.parametrize("cid,batch,num_sms", [(1, 16, 6), (2, 8, 12)])
def test_merge_over_parts(cid, batch, num_sms):
    """Fewer parts than query tokens (6 parts, 16 query tokens of 16 tiles):
    the merge then runs over the parts and visits only the query tokens that
    a part boundary splits; every other token must come out of the decode
    kernel itself.  64 heads and 128 heads."""
    w = synth.make_workload(cid, batch=batch, workers=1)
    dw = DeviceWorkload(w)
    dec = dw.decoder(num_sms)
    assert 1 < dec.num_parts < w.cfg.batch * w.cfg.seq_len_q
    out, lse, err = dw.run(dec=dec)
    assert err == 0
    compare(out, lse, w, all_queries(w))


def test_deterministic():
    w = synth.make_workload(2, batch=2, workers=1)
    dw = DeviceWorkload(w)
    dec = dw.decoder()
    o1, l1, _ = dw.run(dec=dec)
    o1, l1 = o1.clone(), l1.clone()
    o2, l2, _ = dw.run(dec=dec)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_topk1_returns_the_latent():
    rng = np.random.default_rng(12)
    idx = _random_idx(rng, 2, 1, 1, 64)
    w = _custom(16, 1, 64, idx)
    out, lse, _ = DeviceWorkload(w).run()
    for b in range(2):
        g = np.searchsorted(w.ref_pos, idx[b, 0, 0])
        k = oracle.bf16_rne(oracle.dequant_fp8(w.ref_rec[g:g + 1]))[0]
        got = out[b, 0].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.all(got == k[None, :])
    compare(out, lse, w, all_queries(w))


def _off16(shape, dtype, dev):
    """A contiguous tensor starting 16 bytes past a 32-byte boundary."""
    n = math.prod(shape)
    pad = 16 // torch.empty((), dtype=dtype).element_size()
    t = torch.empty(n + pad, dtype=dtype, device=dev)[pad:].view(shape)
    assert int(t.data_ptr()) % 32 == 16
    return t


def test_alignment_paths_agree():
    """q, out and the workspace only 16-byte aligned (the contract's minimum):
    q takes the 128-head kernel's 16-byte load path instead of the 32-byte
    one, and the outputs and split partials leave by TMA stores from either
    base.  Both give the same bits, and both match the oracle (one query
    token's tiles are split over many parts, so the workspace path runs
    too)."""
    w = synth.make_workload(2, batch=1, workers=1)
    dw = DeviceWorkload(w)
    dec = dw.decoder()
    out_a, lse_a, err_a = dw.run(dec=dec)
    assert int(dw.q.data_ptr()) % 32 == 0 and int(out_a.data_ptr()) % 32 == 0
    assert int(dec.workspace.data_ptr()) % 32 == 0
    assert dec.num_parts > 1
    q16 = _off16(tuple(dw.q.shape), torch.bfloat16, dw.dev)
    q16.copy_(dw.q)
    dw.q = q16
    dec.workspace = _off16((dec.workspace.numel(),), torch.uint8, dw.dev)
    out16 = _off16(tuple(out_a.shape), torch.bfloat16, dw.dev)
    dec.error.zero_()
    out_b, lse_b = dec(dw.q, dw.kv, dw.idx, out=out16)
    torch.cuda.synchronize()
    err_b = int(dec.error.item())
    assert out_b.data_ptr() == out16.data_ptr()
    assert err_a == 0 and err_b == 0
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(lse_a, lse_b)
    compare(out_b, lse_b, w, all_queries(w))
