"""Bit-exact dequantization on the GPU (the decode kernel's own routines via
mla_dequantize) against the oracle's decoders rounded once to bf16."""
import numpy as np
import pytest
import torch

import fp4_kv_cache_sparse_gb300 as mla
import oracle
import synth

pytestmark = pytest.mark.gpu


def _gpu_bits(records, fmt):
    t = torch.from_numpy(np.ascontiguousarray(records)).cuda()
    out = mla.dequantize(t, fmt)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def test_fp8_every_data_byte_with_every_scale_byte():
    n = 255
    rec = np.zeros((n, 528), dtype=np.uint8)
    data = (np.arange(512) % 256).astype(np.uint8)
    data[(data & 0x7F) == 0x7F] = 0x00            # NaN codes are outside the contract
    rec[:, :512] = data
    for r in range(n):
        rec[r, 512:] = (r + 17 * np.arange(16)) % 255   # every scale byte 0..254 per block
    want = oracle.bf16_rne(oracle.dequant_fp8(rec))
    got = _gpu_bits(rec, mla.KV_FP8_528)
    assert np.array_equal(got, want), f"{(got != want).sum()} of {got.size} differ"


def test_fp4_every_data_byte_with_every_scale_byte():
    n = 256
    rec = np.zeros((n, 288), dtype=np.uint8)
    rec[:, :256] = np.arange(256, dtype=np.uint8)
    for r in range(n):
        s = (r + 37 * np.arange(32)) % 256
        s[(s & 0x7F) == 0x7F] = 0x38
        rec[r, 256:] = s
    want = oracle.bf16_rne(oracle.dequant_fp4(rec))
    got = _gpu_bits(rec, mla.KV_FP4_288)
    assert np.array_equal(got, want), f"{(got != want).sum()} of {got.size} differ"


@pytest.mark.parametrize("fmt", [mla.KV_FP8_528, mla.KV_FP4_288])
def test_generator_records_exact(fmt):
    rng = np.random.default_rng(3)
    lat = rng.standard_normal((4096, 512), dtype=np.float32) * np.exp(rng.uniform(-8, 8, (4096, 1))).astype(np.float32)
    if fmt == mla.KV_FP8_528:
        rec = synth.encode_fp8_records(lat)
        want = oracle.bf16_rne(oracle.dequant_fp8(rec))
    else:
        rec = synth.encode_fp4_records(lat)
        want = oracle.bf16_rne(oracle.dequant_fp4(rec))
    assert np.array_equal(_gpu_bits(rec, fmt), want)


def test_empty_dequant_is_a_no_op():
    out = mla.dequantize(torch.zeros((0, 528), dtype=torch.uint8, device="cuda"))
    assert out.shape == (0, 512)
