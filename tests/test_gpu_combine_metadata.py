"""GPU split merge (mla_combine) against the oracle's merge, and the
scheduler metadata against the properties a schedule must have (checked
from its own output, not against a copy of the rule that made it)."""
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


def _check_schedule(sched, nsplit, parts, nq, T, max_parts):
    """What "Tile-scheduler metadata" and "split decoding with num_splits"
    ("flops/flashmla-decode-fp8-fp4-kv", "Workarounds") require of the
    schedule, read off the schedule itself:
      - the parts' item ranges [g0, g1) cover 0 .. nq*T once, in order;
      - parts are balanced: every part but the last holds the same number
        of items, the last no more, and there are no more parts than SMs per
        head group;
      - a query token's split count is the number of parts its items fall
        into, and the prefix of those counts is num_splits;
      - a part's first-split id is the number of earlier parts that hold
        items of its first query token, and its first token is g0 // T."""
    G = nq * T
    assert 1 <= parts <= max(max_parts, 1)
    g0, g1 = sched[:, 0].astype(np.int64), sched[:, 1].astype(np.int64)
    assert g0[0] == 0 and g1[-1] == G
    assert np.all(g1 > g0) and np.all(g0[1:] == g1[:-1])
    size = g1 - g0
    assert np.all(size[:-1] == size[0]) and size[-1] <= size[0]
    counts = np.zeros(nq, dtype=np.int64)
    first_local = []
    for k in range(parts):
        qa, qb = g0[k] // T, (g1[k] - 1) // T
        assert sched[k, 3] == qa
        first_local.append(int(counts[qa]))
        counts[qa:qb + 1] += 1
    assert np.array_equal(sched[:, 2], np.array(first_local))
    assert np.array_equal(nsplit, np.concatenate([[0], np.cumsum(counts)]))
    assert np.all(sched[:, 4:] == 0)


@pytest.mark.parametrize("shape", [
    dict(batch=1, seq_len_q=1, h_q=16, topk=64, num_pages=2),
    dict(batch=64, seq_len_q=1, h_q=64, topk=2048, num_pages=64 * 512),
    dict(batch=128, seq_len_q=2, h_q=128, topk=2048, num_pages=128 * 2048),
    dict(batch=32, seq_len_q=1, h_q=16, topk=65536, num_pages=32 * 16384),
    dict(batch=1500, seq_len_q=1, h_q=32, topk=300, num_pages=4),
    dict(batch=64, seq_len_q=1, h_q=64, topk=2048, num_pages=64 * 1024, extra_topk=512, extra_num_pages=64 * 256),
])
@pytest.mark.parametrize("num_sms", [0, 1, 152, 5000])
def test_metadata_is_a_balanced_ordered_partition(shape, num_sms):
    p = mla.Problem.make(**shape)
    sched, nsplit, parts, _ = mla.get_metadata(p, num_sms)
    torch.cuda.synchronize()
    sms = num_sms or torch.cuda.get_device_properties(0).multi_processor_count
    T = math.ceil(p.topk / 128) + math.ceil(p.extra_topk / 128)
    head_groups = p.h_q // min(p.h_q, 64)
    _check_schedule(sched.cpu().numpy().astype(np.int64), nsplit.cpu().numpy().astype(np.int64), parts,
                    p.batch * p.seq_len_q, T, max(sms // head_groups, 1))
