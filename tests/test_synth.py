"""Synthetic workload generator: shapes, index structure, determinism, and
round trips of its encoders through the oracle's decoders.  CPU only."""
import numpy as np
import pytest

import oracle
import synth


@pytest.mark.parametrize("cid", [0, 1, 2, 3, 4, 5, 6])
def test_index_structure(cid):
    cfg = synth.CONFIGS[cid]
    w = synth.make_workload(cid, batch=min(cfg.batch, 2), workers=1)
    b = w.cfg.batch
    assert w.q_bits.shape == (b, cfg.seq_len_q, cfg.h_q, 512)
    assert w.idx.shape == (b, cfg.seq_len_q, cfg.topk)
    for bi in range(b):
        for si in range(cfg.seq_len_q):
            ids = w.idx[bi, si]
            valid = ids[ids >= 0]
            assert np.all(ids[ids < 0] == -1)
            assert (ids == -1).sum() == cfg.neg
            assert len(np.unique(valid)) == len(valid)                       # distinct
            assert np.all((valid >= bi * cfg.pool) & (valid < (bi + 1) * cfg.pool))
            if cfg.neg and cfg.neg_mode == "trailing":
                assert np.all(ids[-cfg.neg:] == -1)
            if cfg.recent_window:
                pos = np.sort(np.concatenate([valid - bi * cfg.pool]))
                recent = (pos >= cfg.pool - cfg.recent_window).sum()
                assert recent >= cfg.topk // 2 - cfg.neg
            if cfg.contiguous:
                assert np.array_equal(ids, bi * cfg.pool + np.arange(cfg.pool - cfg.topk, cfg.pool))
            if cfg.extra_topk:
                x = w.extra_idx[bi, si]
                assert len(np.unique(x)) == cfg.extra_topk
                assert np.all((x >= bi * cfg.extra_pool) & (x < (bi + 1) * cfg.extra_pool))
    # every referenced position has a record
    assert set(np.unique(w.idx[w.idx >= 0]).tolist()) == set(w.ref_pos.tolist())


def test_deterministic_and_worker_independent():
    a = synth.make_workload(3, batch=2, workers=1)
    b = synth.make_workload(3, batch=2, workers=1)
    assert np.array_equal(a.q_bits, b.q_bits) and np.array_equal(a.ref_rec, b.ref_rec)
    assert np.array_equal(a.extra_ref_rec, b.extra_ref_rec)


def test_scattered_neg_moves_the_skips():
    w = synth.make_workload(1, batch=2, scattered_neg=True, workers=1)
    ids = w.idx[0, 0]
    assert (ids == -1).sum() == 20 and not np.all(ids[-20:] == -1)


def test_fp8_encoder_round_trip_error_bound():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((256, 512), dtype=np.float32)
    x[3, :32] = 0.0                                    # an all-zero block
    rec = synth.encode_fp8_records(x)
    dec = oracle.dequant_fp8(rec)
    blocks = np.abs(x.astype(np.float64)).reshape(256, 16, 32).max(axis=2)
    e = rec[:, 512:].astype(np.int64) - 127
    assert np.all(2.0 ** e.astype(float) * 448 >= blocks)             # no saturation needed
    bound = np.maximum(np.abs(x) * 2.0 ** -4, np.repeat(2.0 ** (e - 10).astype(float), 32, axis=1))
    assert np.all(np.abs(dec - x) <= bound)
    assert np.all(dec[3, :32] == 0) and rec[3, 512] == 127


def test_fp4_encoder_round_trip_error_bound():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((256, 512), dtype=np.float32)
    rec = synth.encode_fp4_records(x)
    dec = oracle.dequant_fp4(rec)
    s = np.abs(np.repeat(oracle.dequant_fp4(np.concatenate(
        [np.full((256, 256), 0x22, np.uint8), rec[:, 256:]], axis=1))[:, ::2].reshape(256, 32, 8)[:, :, 0], 16, axis=1))
    amax = np.repeat(np.abs(x).reshape(256, 32, 16).max(axis=2), 16, axis=1)
    assert np.all(np.abs(dec - x) <= s + 0.07 * amax)
    # relative accuracy of the block scale: amax/6 to E4M3 within 2^-4
    assert np.all(np.abs(s * 6 - amax) <= amax * 2.0 ** -4 + 1e-30)


def test_compact_preserves_bytes():
    w = synth.make_workload(1, batch=3, workers=1)
    c = synth.compact(w, [(2, 0), (0, 0)])
    for j, (bi, si) in enumerate([(2, 0), (0, 0)]):
        ids = w.idx[bi, si]
        for t in range(0, ids.shape[0], 97):
            if ids[t] < 0:
                assert c["idx"][j, 0, t] == -1
                continue
            g = np.searchsorted(w.ref_pos, ids[t])
            assert np.array_equal(c["kv"][c["idx"][j, 0, t]], w.ref_rec[g])
