"""Pins of the fp64 oracle against what the pages and mathematics fix.

Nothing here compares the oracle with itself: decoders are checked against
hand-derived bytes and against PyTorch's float8 dtypes, attention against
closed forms, invariants and a library dense-attention routine, the merge
against the unsplit result.  CPU only.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden

D = 512


def _read_cases(name):
    rows = []
    for line in open(golden(name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append(line.split())
    return rows


def _same(a, b):
    """Bitwise-equal doubles (so -0.0 differs from +0.0, NaN equals NaN)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.array_equal(a.view(np.uint64), b.view(np.uint64)) or (
        np.array_equal(np.isnan(a), np.isnan(b))
        and np.array_equal(a[~np.isnan(a)].view(np.uint64), b[~np.isnan(b)].view(np.uint64)))


# --------------------------------------------------------------------------
# Element decoders.
# --------------------------------------------------------------------------

def test_fp8_elements_hand_built():
    for data, scale, expected in _read_cases("fp8_element_cases.txt"):
        rec = np.zeros(528, dtype=np.uint8)
        rec[0] = int(data, 16)
        rec[512] = int(scale)
        got = oracle.dequant_fp8(rec)[0, 0]
        assert _same(got, float(expected)), (data, scale, got, expected)


def test_fp4_elements_hand_built():
    for data, scale, even, odd in _read_cases("fp4_element_cases.txt"):
        rec = np.zeros(288, dtype=np.uint8)
        rec[0] = int(data, 16)
        rec[256] = int(scale, 16)
        got = oracle.dequant_fp4(rec)[0, :2]
        assert _same(got[0], float(even)) and _same(got[1], float(odd)), (data, scale, got)


def test_e4m3fn_all_bytes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3fn(b) for b in range(256)])
    assert _same(got, ref)
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and np.isnan(got).sum() == 2


def test_e8m0_all_bytes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([oracle.e8m0(b) for b in range(256)])
    assert _same(got, ref)
    assert got[127] == 1.0


def test_e2m1_codes_match_ocp_table():
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for code in range(16):
        mag = table[code & 7]
        expected = -mag if code & 8 else mag
        assert _same(oracle.e2m1(code), expected), code


# --------------------------------------------------------------------------
# Record assembly.
# --------------------------------------------------------------------------

def test_fp8_record_scale_block_order():
    # Data 1.0 everywhere, scale byte of block j = 119 + j: dims 32j..32j+31
    # must decode to 2^(j-8).
    rec = np.full(528, 0x38, dtype=np.uint8)
    rec[512:] = 119 + np.arange(16)
    got = oracle.dequant_fp8(rec)[0]
    expected = np.repeat(2.0 ** (np.arange(16) - 8), 32)
    assert np.array_equal(got, expected)


def test_fp8_record_data_order():
    rec = np.zeros(528, dtype=np.uint8)
    rec[:512] = 0x38
    rec[300] = 0x40          # dim 300 alone is 2.0
    rec[512:] = 127
    got = oracle.dequant_fp8(rec)[0]
    assert got[300] == 2.0 and np.count_nonzero(got != 1.0) == 1


def test_fp4_record_nibble_and_scale_order():
    # Byte k holds code 2 (1.0) in the low nibble and code 4 (2.0) in the high
    # nibble: even dims 1.0, odd dims 2.0, times scale block j = 2^(j-16)
    # written as e4m3 (exponent field j - 16 + 7, valid for j >= 10 normal).
    rec = np.zeros(288, dtype=np.uint8)
    rec[:256] = 0x42
    exps = np.arange(32) - 16
    # e4m3 of 2^e for e in [-9, 8]: normal when e >= -6, subnormal below.
    codes = []
    for e in exps:
        e = int(max(min(e, 8), -9))
        codes.append((e + 7) << 3 if e >= -6 else 1 << (e + 9))
    rec[256:] = np.array(codes, dtype=np.uint8)
    got = oracle.dequant_fp4(rec)[0]
    clipped = np.clip(exps, -9, 8)
    scale = np.repeat(2.0 ** clipped, 16)
    base = np.tile([1.0, 2.0], 256)
    assert np.array_equal(got, base * scale)


def test_fp8_random_records_match_torch_decode():
    rng = np.random.default_rng(5)
    recs = rng.integers(0, 256, size=(64, 528), dtype=np.uint8)
    recs[:, :512][(recs[:, :512] & 0x7F) == 0x7F] = 0x38      # no NaN codes
    recs[:, 512:] = rng.integers(100, 150, size=(64, 16))
    elems = torch.from_numpy(recs[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float64)
    scales = torch.from_numpy(recs[:, 512:].copy()).view(torch.float8_e8m0fnu).to(torch.float64)
    ref = (elems.view(64, 16, 32) * scales[:, :, None]).view(64, 512).numpy()
    assert _same(oracle.dequant_fp8(recs), ref)


def test_fp4_random_records_match_table_decode():
    rng = np.random.default_rng(6)
    recs = rng.integers(0, 256, size=(64, 288), dtype=np.uint8)
    sc = recs[:, 256:]
    sc[(sc & 0x7F) == 0x7F] = 0x38
    table = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
    lo = table[recs[:, :256] & 0xF]
    hi = table[recs[:, :256] >> 4]
    vals = np.empty((64, 512))
    vals[:, 0::2] = lo
    vals[:, 1::2] = hi
    scales = torch.from_numpy(recs[:, 256:].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref = vals * np.repeat(scales, 16, axis=1)
    assert _same(oracle.dequant_fp4(recs), ref)


# --------------------------------------------------------------------------
# bfloat16 rounding.
# --------------------------------------------------------------------------

def test_bf16_rne_special_cases():
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0 ** -8, 0x3F80),                  # tie -> even
        (1.0 + 3 * 2.0 ** -8, 0x3F82),              # tie -> even (up)
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),     # above the tie: a float detour would give 0x3F80
        (-0.0, 0x8000),
        (0.0, 0x0000),
        (2.0 ** -133, 0x0001),                      # smallest subnormal
        (2.0 ** -134, 0x0000),                      # tie with zero -> even (0)
        (3 * 2.0 ** -134, 0x0002),                  # tie between 1 and 2 quanta -> 2
        (float(np.finfo(np.float32).max), 0x7F80),  # rounds past the bf16 max
        (3.3895313892515355e38, 0x7F7F),            # bf16 max
        (-448.0, 0xC3E0),
    ]
    for x, bits in cases:
        assert int(oracle.bf16_rne(np.array([x]))[0]) == bits, (x, hex(bits))


def test_bf16_rne_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-60, 60, 100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_rne(x.astype(np.float64)), ref)


# --------------------------------------------------------------------------
# Attention.
# --------------------------------------------------------------------------

def _torch_decode_fp8(recs):
    n = recs.shape[0]
    e = torch.from_numpy(recs[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float64)
    s = torch.from_numpy(recs[:, 512:].copy()).view(torch.float8_e8m0fnu).to(torch.float64)
    return (e.view(n, 16, 32) * s[:, :, None]).view(n, 512)


def _torch_decode_fp4(recs):
    n = recs.shape[0]
    table = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                          -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], dtype=torch.float64)
    b = torch.from_numpy(recs[:, :256].copy()).long()
    v = torch.stack([table[b & 0xF], table[b >> 4]], dim=-1).view(n, 512)
    s = torch.from_numpy(recs[:, 256:].copy()).view(torch.float8_e4m3fn).to(torch.float64)
    return (v.view(n, 32, 16) * s[:, :, None]).view(n, 512)


def _random_fp8_pool(rng, n):
    lat = rng.standard_normal((n, D), dtype=np.float32)
    return synth.encode_fp8_records(lat)


def _q(rng, b, s, h):
    return synth.f32_to_bf16_bits(rng.standard_normal((b, s, h, D), dtype=np.float32))


def _q64(q_bits):
    return oracle.bf16_to_f64(q_bits)


SM = np.float32(1.0 / math.sqrt(D))


def test_topk1_returns_the_latent_exactly():
    rng = np.random.default_rng(11)
    pool = _random_fp8_pool(rng, 8)
    q = _q(rng, 1, 1, 4)
    idx = np.array([[[5, -1, -1]]], dtype=np.int32)
    r = oracle.sparse_mla_decode(q, pool, idx, SM)
    k = _torch_decode_fp8(pool[5:6])[0]
    kb = torch.from_numpy(k.numpy()).to(torch.float32).to(torch.bfloat16)   # k is bf16-exact
    for h in range(4):
        assert np.array_equal(r["out_bf16"][0, 0, h], kb.view(torch.int16).numpy().view(np.uint16))
        x = float(SM) * float(torch.from_numpy(_q64(q[0, 0, h])) @ k)
        assert r["lse"][0, 0, h] == pytest.approx(x, abs=1e-12)


def test_all_skipped_gives_zero_and_neg_inf():
    rng = np.random.default_rng(12)
    pool = _random_fp8_pool(rng, 4)
    q = _q(rng, 2, 1, 3)
    idx = np.full((2, 1, 5), -1, dtype=np.int32)
    r = oracle.sparse_mla_decode(q, pool, idx, SM)
    assert np.all(r["out_bf16"] == 0) and np.all(np.isneginf(r["lse"]))


def test_permutation_invariance():
    rng = np.random.default_rng(13)
    pool = _random_fp8_pool(rng, 96)
    q = _q(rng, 1, 1, 8)
    idx = rng.choice(96, 40, replace=False).astype(np.int32)
    idx[[3, 17]] = -1
    a = oracle.sparse_mla_decode(q, pool, idx[None, None], SM)
    b = oracle.sparse_mla_decode(q, pool, rng.permutation(idx)[None, None], SM)
    np.testing.assert_allclose(a["out_f64"], b["out_f64"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=0, atol=1e-12)
    diff = np.abs(a["out_bf16"].astype(np.int32) - b["out_bf16"].astype(np.int32))
    assert diff.max() <= 1


def test_duplicate_token_adds_ln2():
    rng = np.random.default_rng(14)
    pool = _random_fp8_pool(rng, 6)
    q = _q(rng, 1, 1, 5)
    one = oracle.sparse_mla_decode(q, pool, np.array([[[2]]], np.int32), SM)
    two = oracle.sparse_mla_decode(q, pool, np.array([[[2, 2]]], np.int32), SM)
    assert np.array_equal(one["out_bf16"], two["out_bf16"])
    np.testing.assert_allclose(two["lse"], one["lse"] + math.log(2.0), atol=1e-12)


def test_zero_query_gives_mean_and_log_n():
    rng = np.random.default_rng(15)
    pool = _random_fp8_pool(rng, 20)
    q = np.zeros((1, 1, 2, D), dtype=np.uint16)
    ids = np.array([1, 4, 7, 9, 15, 19, -1], dtype=np.int32)
    r = oracle.sparse_mla_decode(q, pool, ids[None, None], SM)
    k = _torch_decode_fp8(pool[ids[ids >= 0]]).numpy()
    np.testing.assert_allclose(r["out_f64"][0, 0, 0], k.mean(axis=0), rtol=1e-13, atol=1e-15)
    assert r["lse"][0, 0, 1] == pytest.approx(math.log(6.0), abs=1e-13)


def test_brute_force_dense_attention_fp8():
    """Indices = the whole pool: the result must be library dense attention
    (scaled_dot_product_attention in fp64) with K = V = decoded latents."""
    rng = np.random.default_rng(16)
    n = 128
    pool = _random_fp8_pool(rng, n)
    b, h = 2, 16
    q = _q(rng, b, 1, h)
    idx = np.stack([rng.permutation(n) for _ in range(b)]).astype(np.int32)[:, None]
    r = oracle.sparse_mla_decode(q, pool, idx, SM)
    K = _torch_decode_fp8(pool)
    for bi in range(b):
        Q = torch.from_numpy(_q64(q[bi, 0]))                       # [h, 512]
        o = torch.nn.functional.scaled_dot_product_attention(
            Q[None, :, None, :], K[None, None], K[None, None], scale=float(SM))[0, :, 0, :]
        np.testing.assert_allclose(r["out_f64"][bi, 0], o.numpy(), rtol=1e-10, atol=1e-12)
        lse = torch.logsumexp((Q @ K.T) * float(SM), dim=-1)
        np.testing.assert_allclose(r["lse"][bi, 0], lse.numpy(), rtol=0, atol=1e-10)


def test_brute_force_joint_softmax_fp8_plus_fp4():
    """Main + extra cache under one softmax == dense attention over the
    concatenation of both decoded token sets."""
    rng = np.random.default_rng(17)
    pool = _random_fp8_pool(rng, 64)
    xpool = synth.encode_fp4_records(rng.standard_normal((32, D), dtype=np.float32))
    q = _q(rng, 1, 1, 16)
    idx = rng.choice(64, 24, replace=False).astype(np.int32)
    xidx = rng.choice(32, 10, replace=False).astype(np.int32)
    xidx[4] = -1
    r = oracle.sparse_mla_decode(q, pool, idx[None, None], SM, extra_kv=xpool, extra_idx=xidx[None, None])
    K = torch.cat([_torch_decode_fp8(pool[idx]), _torch_decode_fp4(xpool[xidx[xidx >= 0]])])
    Q = torch.from_numpy(_q64(q[0, 0]))
    o = torch.nn.functional.scaled_dot_product_attention(
        Q[None, :, None, :], K[None, None], K[None, None], scale=float(SM))[0, :, 0, :]
    np.testing.assert_allclose(r["out_f64"][0, 0], o.numpy(), rtol=1e-10, atol=1e-12)
    lse = torch.logsumexp((Q @ K.T) * float(SM), dim=-1)
    np.testing.assert_allclose(r["lse"][0, 0], lse.numpy(), atol=1e-10)


def test_out_of_range_indices_are_skipped_and_counted():
    rng = np.random.default_rng(18)
    pool = _random_fp8_pool(rng, 10)
    q = _q(rng, 1, 1, 2)
    good = oracle.sparse_mla_decode(q, pool, np.array([[[1, 3, -1]]], np.int32), SM)
    bad = oracle.sparse_mla_decode(q, pool, np.array([[[1, 3, 10, -7, -1]]], np.int32), SM)
    assert bad["bad"] == 2 and good["bad"] == 0
    assert np.array_equal(good["out_bf16"], bad["out_bf16"])


# --------------------------------------------------------------------------
# Split merge.
# --------------------------------------------------------------------------

def test_combine_over_any_partition_equals_unsplit():
    rng = np.random.default_rng(19)
    pool = _random_fp8_pool(rng, 200)
    q = _q(rng, 1, 1, 8)
    ids = rng.choice(200, 120, replace=False).astype(np.int32)
    full = oracle.sparse_mla_decode(q, pool, ids[None, None], SM)
    cuts = [0, 7, 50, 51, 120]
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sub = np.full_like(ids, -1)
        sub[a:b] = ids[a:b]
        r = oracle.sparse_mla_decode(q, pool, sub[None, None], SM)
        parts_o.append(r["out_f64"].reshape(8, D))
        parts_l.append(r["lse"].reshape(8))
    # An empty split (all -1) must weigh nothing.
    e = oracle.sparse_mla_decode(q, pool, np.full((1, 1, 4), -1, np.int32), SM)
    parts_o.append(e["out_f64"].reshape(8, D))
    parts_l.append(e["lse"].reshape(8))
    o, l = oracle.combine(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(o, full["out_f64"].reshape(8, D), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(l, full["lse"].reshape(8), atol=1e-12)


def test_combine_single_split_is_identity_and_all_empty_is_zero():
    rng = np.random.default_rng(20)
    o = rng.standard_normal((1, 3, D))
    l = rng.standard_normal((1, 3))
    out, lse = oracle.combine(o, l)
    np.testing.assert_allclose(out, o[0], rtol=1e-15)
    np.testing.assert_allclose(lse, l[0], rtol=1e-15)
    out, lse = oracle.combine(o[[0, 0]] * 0 + 5.0, np.full((2, 3), -np.inf))
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_joint_softmax_is_the_merge_of_main_and_extra():
    rng = np.random.default_rng(21)
    pool = _random_fp8_pool(rng, 50)
    xpool = synth.encode_fp4_records(rng.standard_normal((30, D), dtype=np.float32))
    q = _q(rng, 1, 1, 4)
    idx = rng.choice(50, 20, replace=False).astype(np.int32)[None, None]
    xidx = rng.choice(30, 9, replace=False).astype(np.int32)[None, None]
    joint = oracle.sparse_mla_decode(q, pool, idx, SM, extra_kv=xpool, extra_idx=xidx)
    main = oracle.sparse_mla_decode(q, pool, idx, SM)
    extra = oracle.sparse_mla_decode(q, pool, np.full_like(idx, -1), SM, extra_kv=xpool, extra_idx=xidx)
    o, l = oracle.combine(np.stack([main["out_f64"].reshape(4, D), extra["out_f64"].reshape(4, D)]),
                          np.stack([main["lse"].reshape(4), extra["lse"].reshape(4)]))
    np.testing.assert_allclose(o, joint["out_f64"].reshape(4, D), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(l, joint["lse"].reshape(4), atol=1e-12)


# --------------------------------------------------------------------------
# Record encoders (the KV-cache writer's quantizer).
# --------------------------------------------------------------------------

def _e4m3_values():
    return np.array([oracle.e4m3fn(c) for c in range(0x7F)])  # finite non-negative codes


def test_e4m3fn_rne_round_trips_every_code_and_matches_torch():
    """Every finite code decodes and re-encodes to itself (both signs); on
    random in-range values the nearest-even rounding agrees with PyTorch's
    float64 -> float8_e4m3fn conversion."""
    for c in list(range(0x7F)) + [0x80 | c for c in range(0x7F)]:
        assert oracle.e4m3fn_rne(oracle.e4m3fn(c)) == c
    rng = np.random.default_rng(5)
    x = rng.uniform(-448, 448, 4000) * 2.0 ** rng.integers(-12, 1, 4000)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3fn_rne(v) for v in x], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_e4m3fn_rne_ties_go_to_the_even_code_and_saturate():
    vals = _e4m3_values()
    for c in range(0x7E):
        mid = (vals[c] + vals[c + 1]) / 2.0
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3fn_rne(mid) == even
        assert oracle.e4m3fn_rne(-mid) == 0x80 | even
    assert oracle.e4m3fn_rne(448.0) == 0x7E
    assert oracle.e4m3fn_rne(1e30) == 0x7E
    assert oracle.e4m3fn_rne(-1e30) == 0xFE
    assert oracle.e4m3fn_rne(-0.0) == 0x80


def test_e2m1_rne_codes_ties_and_saturation():
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c, v in enumerate(grid):
        assert oracle.e2m1_rne(v) == c and oracle.e2m1_rne(-v) == 8 | c
    for c in range(7):
        mid = (grid[c] + grid[c + 1]) / 2.0
        assert oracle.e2m1_rne(mid) == (c if c % 2 == 0 else c + 1)
    assert oracle.e2m1_rne(7.0) == 7 and oracle.e2m1_rne(100.0) == 7 and oracle.e2m1_rne(-9.0) == 15


def _fp8_records_with_full_blocks(rng, n):
    """Random FP8 records whose every block holds a +-448 code (0x7E/0xFE),
    so that the block maximum fixes the scale."""
    rec = rng.integers(0, 256, (n, 528)).astype(np.uint8)
    data = rec[:, :512]
    data[(data & 0x7F) == 0x7F] ^= 0x01          # no NaN codes
    for b in range(16):
        pos = 32 * b + rng.integers(0, 32, n)
        data[np.arange(n), pos] = np.where(rng.random(n) < 0.5, 0x7E, 0xFE)
    rec[:, 512:] = rng.integers(100, 150, (n, 16))
    return rec


def test_encode_fp8_inverts_decode_when_the_maximum_is_448():
    rng = np.random.default_rng(6)
    rec = _fp8_records_with_full_blocks(rng, 64)
    assert np.array_equal(oracle.encode_fp8(oracle.dequant_fp8(rec)), rec)


def test_encode_fp8_scale_is_the_least_power_of_two_and_rounding_is_within_half_a_step():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((50, 512)) * 2.0 ** rng.integers(-20, 20, (50, 1))
    x[3, 32:64] = 0.0                          # an all-zero block
    rec = oracle.encode_fp8(x)
    e = rec[:, 512:].astype(np.int64) - 127
    amax = np.abs(x.reshape(50, 16, 32)).max(axis=2)
    nz = amax > 0
    assert np.all(amax[nz] * 2.0 ** -e[nz] <= 448.0)
    assert np.all(amax[nz] * 2.0 ** -(e[nz] - 1) > 448.0)
    assert rec[3, 513] == 127                  # zero block: scale 1
    assert np.all((rec[3, 32:64] & 0x7F) == 0)
    # |decode(encode(x)) - x| <= half the E4M3 step at the scaled value's binade.
    y = x * 2.0 ** -np.repeat(e, 32, axis=1)
    binade = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6)))
    half_step = 2.0 ** (binade - 4) * 2.0 ** np.repeat(e, 32, axis=1)
    err = np.abs(oracle.dequant_fp8(rec) - x)
    assert np.all(err <= half_step * (1 + 1e-12))


def test_encode_fp4_inverts_decode_when_a_block_holds_6():
    rng = np.random.default_rng(8)
    n = 40
    rec = rng.integers(0, 256, (n, 288)).astype(np.uint8)
    # Scales: finite, non-zero E4M3 codes whose value times 6 stays exact.
    rec[:, 256:] = rng.integers(0x20, 0x60, (n, 32))
    codes = np.stack([rec[:, :256] & 0xF, rec[:, :256] >> 4], axis=2).reshape(n, 512)
    for b in range(32):
        pos = 16 * b + rng.integers(0, 16, n)
        codes[np.arange(n), pos] = np.where(rng.random(n) < 0.5, 0x7, 0xF)
    codes[codes == 0x8] = 0x0                  # -0 and +0 decode alike; keep +0
    rec[:, :256] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(oracle.encode_fp4(oracle.dequant_fp4(rec)), rec)


def test_encoders_agree_with_the_test_input_quantizer():
    """The harness quantizer (numpy, its own code) and the oracle (C, a scan
    over codes) apply the same rule to bf16-valued inputs."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((30, 512)).astype(np.float32) * 2.0 ** rng.integers(-10, 10, (30, 1)).astype(np.float32)
    x = oracle.bf16_to_f64(synth.f32_to_bf16_bits(x)).astype(np.float32)
    assert np.array_equal(oracle.encode_fp8(x), synth.encode_fp8_records(x))
    assert np.array_equal(oracle.encode_fp4(x), synth.encode_fp4_records(x))


# --------------------------------------------------------------------------
# Output-side epilogue: conjugate rotary embedding of dims 448..511 and the
# FP8 cast ("deepseek-ai/FlashMLA", "What it is"; qk_rope_head_dim = 64 on
# "flops/attn-mla-kernel-support-matrix", "notes").  Which dims, the pairing
# and the frequency rule are readings; these pins check that what is built
# is a rotation with the stated convention, not the arithmetic retyped.
# --------------------------------------------------------------------------

THETA = 10000.0


def _rows(n, seed):
    return np.random.default_rng(seed).standard_normal((n, D))


def test_rope_position_zero_is_the_identity():
    x = _rows(6, 1)
    assert _same(oracle.rope_rotate(x, np.zeros(6, dtype=np.int64), THETA, -1), x)
    recs = oracle.rope_fp8_epilogue(x, np.zeros(6, dtype=np.int64), THETA)
    assert np.array_equal(recs, oracle.encode_fp8(x))


def test_rope_conjugate_undoes_the_forward_rotation_and_keeps_pair_norms():
    x = _rows(8, 2)
    pos = np.array([1, 17, 4095, 65536, 131071, 7, 0, 100000])
    y = oracle.rope_rotate(x, pos, THETA, -1)
    back = oracle.rope_rotate(y, pos, THETA, +1)
    assert np.abs(back - x).max() < 1e-12
    assert _same(y[:, :448], x[:, :448])               # only the last 64 dims turn
    nx = np.hypot(x[:, 448::2], x[:, 449::2])
    ny = np.hypot(y[:, 448::2], y[:, 449::2])
    assert np.abs(nx - ny).max() < 1e-12               # each pair is rotated, not scaled


def test_rope_angles_add():
    """Turning by position p1 and then p2 is turning by p1 + p2 (what makes
    it a rotary position encoding); a sign slip in one term breaks this."""
    x = _rows(4, 3)
    p1, p2 = np.array([3, 100, 2048, 9]), np.array([5, 28, 999, 40000])
    two = oracle.rope_rotate(oracle.rope_rotate(x, p1, THETA, -1), p2, THETA, -1)
    one = oracle.rope_rotate(x, p1 + p2, THETA, -1)
    assert np.abs(two - one).max() < 1e-9


def test_rope_frequencies_of_pairs_0_and_16():
    """Pair 0 turns by pos radians (theta^0 = 1); pair 16 by pos * theta^-1/2,
    i.e. 1 radian at pos 100 for theta = 10^4; the conjugate side turns
    clockwise: (1, 0) -> (cos phi, -sin phi)."""
    x = np.zeros((2, D))
    x[:, 448] = 1.0            # pair 0
    x[:, 448 + 32] = 1.0       # pair 16
    y = oracle.rope_rotate(x, np.array([1, 100]), THETA, -1)
    assert abs(y[0, 448] - math.cos(1.0)) < 1e-15 and abs(y[0, 449] + math.sin(1.0)) < 1e-15
    assert abs(y[1, 480] - math.cos(1.0)) < 1e-12 and abs(y[1, 481] + math.sin(1.0)) < 1e-12


def test_rope_fp8_records_decode_to_the_rotated_rows_within_one_step():
    x = _rows(16, 4) * np.logspace(-3, 3, 16)[:, None]
    pos = np.arange(16) * 977
    recs = oracle.rope_fp8_epilogue(x, pos, THETA)
    y = oracle.rope_rotate(x, pos, THETA, -1)
    got = oracle.dequant_fp8(recs.reshape(-1, 528)).reshape(y.shape)
    # Per 32-value block the scale is the least power of two 2^e bringing the
    # block maximum within 448; an e4m3 value then lies within half a step
    # (2^(floor(log2|v|) - 4), at least 2^-10 in scaled units) of the input.
    for r in range(16):
        for blk in range(16):
            v = y[r, 32 * blk:32 * blk + 32]
            e = int(recs[r, 512 + blk]) - 127
            s = np.abs(v) * 2.0 ** -e
            half = np.where(s > 0, 2.0 ** (np.floor(np.log2(np.maximum(s, 1e-300))) - 4), 0)
            half = np.maximum(half, 2.0 ** -10)
            assert np.all(np.abs(got[r, 32 * blk:32 * blk + 32] * 2.0 ** -e - v * 2.0 ** -e) <= half + 1e-15)
