"""GPU split merge (mla_combine) against the oracle's merge, and the
scheduler metadata against a restatement of its partition rule."""
import math

import numpy as np
import pytest
import torch

import fp4_kv_cache_sparse_gb300 as mla
import oracle

pytestmark = pytest.mark.gpu


def test_combine_matches_oracle_merge():
    rng = np.random.default_rng(1)
    h = 16
    counts = [1, 3, 2, 1, 4, 2]
    nq = len(counts)
    prefix = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    total = int(prefix[-1])
    o = rng.standard_normal((total, h, 512)).astype(np.float32)
    l = (rng.standard_normal((total, h)) * 5).astype(np.float32)
    l[1, 3] = -np.inf                          # an empty split inside a query
    l[prefix[5]:prefix[6]] = -np.inf           # a query whose splits are all empty
    p = mla.Problem.make(nq, 1, h, 128, 4)
    out = torch.empty((nq, 1, h, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((nq, 1, h), dtype=torch.float32, device="cuda")
    mla.combine(p, torch.from_numpy(prefix).cuda(), torch.from_numpy(o).cuda(), torch.from_numpy(l).cuda(),
                out, lse)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()[:, 0].astype(np.float64)
    gl = lse.cpu().numpy()[:, 0].astype(np.float64)
    for q in range(nq):
        a, b = prefix[q], prefix[q + 1]
        ro, rl = oracle.combine(o[a:b].astype(np.float64), l[a:b].astype(np.float64))
        want = oracle.bf16_to_f64(oracle.bf16_rne(ro))
        assert np.all(np.abs(got[q] - want) <= 1e-2 + 1e-2 * np.abs(want))
        both = np.isneginf(gl[q]) & np.isneginf(rl)
        assert np.all(both | (np.abs(gl[q] - rl) <= 1e-3))
    assert np.all(got[5] == 0) and np.all(np.isneginf(gl[5]))


def _restated(p, num_sms):
    nh = min(p.h_q, 64)
    T = math.ceil(p.topk / 128) + math.ceil(p.extra_topk / 128)
    nq = p.batch * p.seq_len_q
    G = nq * T
    target = min(max(num_sms // (p.h_q // nh), 1), G)
    S = math.ceil(G / target)
    parts = math.ceil(G / S)
    sched = []
    for k in range(parts):
        g0, g1 = k * S, min(G, (k + 1) * S)
        q0 = g0 // T
        sched.append([g0, g1, k - (q0 * T) // S, q0, 0, 0, 0, 0])
    splits = [((q + 1) * T - 1) // S - (q * T) // S + 1 for q in range(nq)]
    return np.array(sched, np.int32), np.concatenate([[0], np.cumsum(splits)]).astype(np.int32)


@pytest.mark.parametrize("shape", [
    dict(batch=1, seq_len_q=1, h_q=16, topk=64, num_pages=2),
    dict(batch=64, seq_len_q=1, h_q=64, topk=2048, num_pages=64 * 512),
    dict(batch=128, seq_len_q=2, h_q=128, topk=2048, num_pages=128 * 2048),
    dict(batch=32, seq_len_q=1, h_q=16, topk=65536, num_pages=32 * 16384),
    dict(batch=1500, seq_len_q=1, h_q=32, topk=300, num_pages=4),
])
@pytest.mark.parametrize("num_sms", [0, 1, 152, 5000])
def test_metadata_matches_partition_rule(shape, num_sms):
    p = mla.Problem.make(**shape)
    sched, nsplit, parts, _ = mla.get_metadata(p, num_sms)
    torch.cuda.synchronize()
    sms = num_sms or torch.cuda.get_device_properties(0).multi_processor_count
    rs, rn = _restated(p, sms)
    assert parts == rs.shape[0]
    assert np.array_equal(sched.cpu().numpy(), rs)
    assert np.array_equal(nsplit.cpu().numpy(), rn)
