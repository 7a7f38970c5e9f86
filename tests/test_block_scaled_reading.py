"""The block-scaled QK^T question ("flops/flashmla-decode-fp8-fp4-kv",
"Workarounds": per-token inlined scales "so dequant is free in the attention
kernel"; "Arithmetic intensity": one e8m0 scale per 32 values).  A
block-scaled (MX) product would take K's e4m3 bytes and e8m0 scales as they
are stored and needs Q in the same form: Q quantized per 32 values with the
writer's scale rule.  These tests measure, with the oracle's own encoder and
decoders, what that does to the result against the decode tolerances
(lse within 1e-3): one e4m3 level of Q breaks the bound; a hi + lo pair
(the residual quantized again) stays far inside it.  CPU only."""
import numpy as np

import oracle
import synth


def _mx(x):
    """Rows of 512 values as the writer would store them (e4m3 per 32
    values under an e8m0 power-of-two scale), decoded back."""
    rows = x.reshape(-1, 512)
    return oracle.dequant_fp8(oracle.encode_fp8(rows)).reshape(x.shape)


def _lse_errors(cid, n):
    w = synth.make_workload(cid, batch=min(n, 8), workers=1)
    qs = [(b, 0) for b in range(min(n, w.cfg.batch))]
    c = synth.compact(w, qs)
    K = oracle.dequant_fp8(c["kv"])
    q = oracle.bf16_to_f64(c["q_bits"])[:, 0]               # [n, h, 512]
    q_hi = _mx(q)
    q_lo = _mx(q - q_hi)
    scale = float(np.float32(w.sm_scale))
    one, two = [], []
    ref = oracle.sparse_mla_decode(c["q_bits"], c["kv"], c["idx"], w.sm_scale)["lse"][:, 0]
    for j in range(len(qs)):
        ids = c["idx"][j, 0]
        Ks = K[ids[ids >= 0]]

        def lse(qq):
            s = qq @ Ks.T * scale
            m = s.max(-1, keepdims=True)
            return (m + np.log(np.exp(s - m).sum(-1, keepdims=True)))[:, 0]

        one.append(np.abs(lse(q_hi[j]) - ref[j]).max())
        two.append(np.abs(lse(q_hi[j] + q_lo[j]) - ref[j]).max())
    return max(one), max(two)


def test_single_level_q_breaks_the_lse_bound_and_hi_lo_does_not():
    for cid, n in ((0, 1), (1, 4)):
        one, two = _lse_errors(cid, n)
        assert one > 1e-3, (cid, one)        # one e4m3 level of Q: outside the bound
        assert two < 1e-6, (cid, two)        # hi + lo: far inside it
