"""GPU KV-cache writer (mla_kv_write) against the oracle's record encoders,
byte for byte: the records it stores, the records it leaves alone, and the
slots it refuses."""
import numpy as np
import pytest
import torch

import fp4_kv_cache_sparse_gb300 as mla
import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
REC = {mla.KV_FP8_528: 528, mla.KV_FP4_288: 288}
ENCODE = {mla.KV_FP8_528: oracle.encode_fp8, mla.KV_FP4_288: oracle.encode_fp4}


def _latents(n, seed):
    """bf16 latents with the awkward cases: per-token magnitudes over many
    binades, all-zero blocks, negative zeros, tiny and large values, ties."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 512)).astype(np.float32)
    x *= (2.0 ** rng.integers(-30, 30, (n, 1))).astype(np.float32)
    x[0, :32] = 0.0                              # an all-zero FP8 block
    x[0, 32:48] = -0.0                           # negative zeros
    x[1, :] = 448.0 * 2.0 ** -3                  # exact grid values
    x[2, :16] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 2, dtype=np.float32)  # e2m1 ties at s = 1
    x[3, :] = 3.0e4 * rng.standard_normal(512).astype(np.float32)  # FP4 scale saturates at 448
    x[4, :] = 1.0e-30 * rng.standard_normal(512).astype(np.float32)  # tiny values
    bits = synth.f32_to_bf16_bits(x)
    return bits, oracle.bf16_to_f64(bits)


def _pool(kv_format, tokens):
    return torch.full((tokens, REC[kv_format]), synth.POISON_BYTE, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("kv_format", [mla.KV_FP8_528, mla.KV_FP4_288])
def test_writer_matches_the_oracle_encoder_byte_for_byte(kv_format):
    n, tokens = 300, 64 * 16
    bits, x = _latents(n, 31 + kv_format)
    rng = np.random.default_rng(7)
    slots = rng.choice(tokens, n, replace=False).astype(np.int32)
    pool = _pool(kv_format, tokens)
    lat = torch.from_numpy(bits.view(np.int16)).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.kv_write(lat, torch.from_numpy(slots).to(DEV), pool, kv_format, error=err)
    torch.cuda.synchronize()
    got = pool.cpu().numpy()
    want = ENCODE[kv_format](x)
    assert int(err.item()) == 0
    for t in range(n):
        assert np.array_equal(got[slots[t]], want[t]), f"token {t}: first differing byte " \
            f"{int(np.nonzero(got[slots[t]] != want[t])[0][0])}"
    untouched = np.setdiff1d(np.arange(tokens), slots)
    assert np.all(got[untouched] == synth.POISON_BYTE)


@pytest.mark.parametrize("kv_format", [mla.KV_FP8_528, mla.KV_FP4_288])
def test_writer_skips_minus_one_and_flags_bad_slots(kv_format):
    n, pages = 6, 2
    bits, x = _latents(n, 5)
    slots = np.array([3, -1, 127, 128, -7, 64], dtype=np.int32)  # 128 = 2 pages * 64: out of range
    pool = _pool(kv_format, pages * 64)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.kv_write(torch.from_numpy(bits.view(np.int16)).to(DEV), torch.from_numpy(slots).to(DEV), pool, kv_format,
                 num_pages=pages, error=err)
    torch.cuda.synchronize()
    got = pool.cpu().numpy()
    want = ENCODE[kv_format](x)
    assert int(err.item()) & mla.DEVERR_BAD_INDEX
    for t in (0, 2, 5):
        assert np.array_equal(got[slots[t]], want[t])
    written = {3, 127, 64}
    assert all(np.all(got[r] == synth.POISON_BYTE) for r in range(pages * 64) if r not in written)


def test_written_records_decode_as_the_decode_kernel_reads_them():
    """Write, then read back through the decode kernel's own dequantizer: the
    values are the oracle's decoding of the oracle's encoding."""
    n = 64
    bits, x = _latents(n, 9)
    for kv_format, dec in ((mla.KV_FP8_528, oracle.dequant_fp8), (mla.KV_FP4_288, oracle.dequant_fp4)):
        pool = _pool(kv_format, n)
        mla.kv_write(torch.from_numpy(bits.view(np.int16)).to(DEV),
                     torch.arange(n, dtype=torch.int32, device=DEV), pool, kv_format)
        got = mla.dequantize(pool, kv_format).view(torch.int16).cpu().numpy().view(np.uint16)
        want = oracle.bf16_rne(dec(ENCODE[kv_format](x)))
        assert np.array_equal(got, want)
