"""Shared helpers of the GPU parity tests: device pools from a synthetic
workload, a decode through the C ABI, and the oracle on sampled query
tokens.  (Test infrastructure.)"""
import numpy as np
import torch

import fp4_kv_cache_sparse_gb300 as mla
import oracle
import synth

OUT_ATOL = 1e-2      # |err| <= 1e-2 + 1e-2 |ref| on bf16 outputs
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3      # absolute, natural log


def device_pool(pos, rec, tokens, dev, poison=synth.POISON_BYTE):
    R = rec.shape[1]
    pool = torch.full((tokens, R), poison, dtype=torch.uint8, device=dev)
    if pos.shape[0]:
        pool[torch.from_numpy(pos).to(dev)] = torch.from_numpy(rec).to(dev)
    return pool


class DeviceWorkload:
    def __init__(self, w: synth.Workload, dev=None):
        dev = dev or torch.device("cuda", 0)
        self.w = w
        self.dev = dev
        self.q = torch.from_numpy(w.q_bits.view(np.int16)).to(dev).view(torch.bfloat16)
        self.idx = torch.from_numpy(w.idx).to(dev)
        self.kv = device_pool(w.ref_pos, w.ref_rec, w.pool_tokens, dev)
        self.xkv = self.xidx = None
        if w.extra_idx is not None:
            self.xkv = device_pool(w.extra_ref_pos, w.extra_ref_rec, w.extra_pool_tokens, dev)
            self.xidx = torch.from_numpy(w.extra_idx).to(dev)
        c = w.cfg
        self.problem = mla.Problem.make(
            c.batch, c.seq_len_q, c.h_q, c.topk, w.pool_tokens // 64,
            extra_topk=c.extra_topk, extra_num_pages=w.extra_pool_tokens // 64, sm_scale=float(w.sm_scale))

    def decoder(self, num_sms=0):
        return mla.SparseMLADecoder(self.problem, self.dev, num_sms=num_sms)

    def run(self, num_sms=0, dec=None):
        dec = dec or self.decoder(num_sms)
        dec.error.zero_()
        out, lse = dec(self.q, self.kv, self.idx, self.xkv, self.xidx)
        torch.cuda.synchronize()
        return out, lse, int(dec.error.item())


def oracle_on(w: synth.Workload, queries):
    c = synth.compact(w, queries)
    return oracle.sparse_mla_decode(c["q_bits"], c["kv"], c["idx"], w.sm_scale,
                                    extra_kv=c.get("extra_kv"), extra_idx=c.get("extra_idx"))


def compare(out, lse, w, queries, ref=None):
    """Element-wise check of the GPU result on the given (b, s) query tokens."""
    ref = ref or oracle_on(w, queries)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    for j, (bi, si) in enumerate(queries):
        got = o[bi, si].astype(np.float64)
        want = oracle.bf16_to_f64(ref["out_bf16"][j, 0])
        err = np.abs(got - want)
        bad = err > OUT_ATOL + OUT_RTOL * np.abs(want)
        assert not bad.any(), f"query {(bi, si)}: {bad.sum()} outputs off, max err {err.max():.4g}"
        gl, wl = l[bi, si].astype(np.float64), ref["lse"][j, 0]
        both_inf = np.isneginf(gl) & np.isneginf(wl)
        lerr = np.where(both_inf, 0.0, np.abs(gl - wl))
        assert np.all(lerr <= LSE_ATOL), f"query {(bi, si)}: max lse err {np.nanmax(lerr):.4g}"
    return ref


def all_queries(w):
    return [(b, s) for b in range(w.cfg.batch) for s in range(w.cfg.seq_len_q)]


def sample_queries(w, n=4, seed=0):
    qs = all_queries(w)
    rng = np.random.default_rng(seed)
    pick = sorted(set([0, len(qs) - 1] + list(rng.choice(len(qs), min(n, len(qs)), replace=False))))
    return [qs[i] for i in pick]
