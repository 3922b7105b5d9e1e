"""Pins for the oracle's MXFP8 quantizer (no GPU): hand-worked blocks, the closed form of the
round-up E8M0 rule over every bf16 magnitude, and the independence of the columnwise copy."""
import numpy as np
import pytest
import torch

import oracle
from tests._golden import hexbytes, load


@pytest.mark.parametrize("blk", load("mxfp8_blocks.json")["blocks"], ids=lambda b: b["name"])
def test_hand_worked_blocks(blk):
    bits = np.zeros(32, dtype=np.uint16)
    given = np.array([int(b, 16) for b in blk["bf16_bits"]], dtype=np.uint16)
    bits[:len(given)] = given
    out = oracle.mxfp8_quantize(bits.reshape(1, 32), rowwise=True, colwise=False)
    assert out["sf_row"][0, 0] == int(blk["sf"], 16)
    want = np.zeros(32, dtype=np.uint8)
    want[:len(blk["codes"])] = hexbytes(blk["codes"])
    assert np.array_equal(out["q_row"][0], want)


def _all_positive_bf16():
    bits = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)   # +min subnormal .. +max
    return bits, oracle.bf16_bits_to_f64(bits)


def test_e8m0_round_up_closed_form_exhaustive():
    # For every positive finite bf16 amax: never clipped (amax * 2^-e <= 448), and minimal
    # (amax * 2^-e > 224, i.e. e-1 would clip) unless the E8M0 floor 2^-127 was hit.
    _, a = _all_positive_bf16()
    e = oracle.e8m0_exponent(a)
    scaled = np.ldexp(a, -e)
    assert np.all(scaled <= 448.0)
    free = e > -127
    assert np.all(scaled[free] > 224.0)
    assert np.all(a[~free] <= 448.0 * 2.0 ** -127)
    assert oracle.e8m0_exponent(np.array([0.0]))[0] == -127


def test_e8m0_exponent_equals_log2_ceiling():
    # Independent closed form on exactly representable ratios: amax = 448 * 2^k * (1 + f).
    for k in range(-120, 120, 7):
        assert oracle.e8m0_exponent(np.array([448.0 * 2.0 ** k]))[0] == k
        assert oracle.e8m0_exponent(np.array([448.0 * 2.0 ** k * (1 + 2 ** -20)]))[0] == k + 1
        assert oracle.e8m0_exponent(np.array([224.0 * 2.0 ** k * (1 + 2 ** -20)]))[0] == k


def test_block_amax_code_lies_in_224_to_448():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-20, 20, (64, 1)))).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out = oracle.mxfp8_quantize(bits, colwise=False)
    q = out["q_row"].reshape(64, 8, 32)
    mag = q & 0x7F
    # the scaled block amax lies in (224, 448], so its code is 224 (0x76) .. 448 (0x7E) whenever
    # e > -127: never saturated, never more than one binade below the top
    top = mag.max(axis=2)
    assert np.all((top >= 0x76) & (top <= 0x7E))


def test_columnwise_is_rowwise_of_transpose():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 96)).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    both = oracle.mxfp8_quantize(bits)
    rowT = oracle.mxfp8_quantize(np.ascontiguousarray(bits.T), colwise=False)
    assert np.array_equal(both["q_colT"], rowT["q_row"])
    assert np.array_equal(both["sf_colT"], rowT["sf_row"])


def test_columnwise_differs_from_requantizing_rowwise_copy():
    # The pages: rowwise and columnwise blocks are numerically different and must each come from
    # the full-precision data. Requantizing the dequantized rowwise copy along columns is not the
    # same thing; show that it changes bytes on ordinary data.
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((128, 128)) * np.exp(rng.uniform(-3, 3, (128, 1)))).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    direct = oracle.mxfp8_quantize(bits)
    deq = oracle.dequantize_mxfp8(direct["q_row"], direct["sf_row"])
    requant = oracle.mxfp8_quantize(deq, rowwise=False)
    assert not np.array_equal(requant["q_colT"], direct["q_colT"])


def test_zeros_and_maxes_families():
    z = np.zeros((32, 64), dtype=np.uint16)
    out = oracle.mxfp8_quantize(z)
    assert not out["q_row"].any() and not out["sf_row"].any()
    assert not out["q_colT"].any() and not out["sf_colT"].any()
    m = np.full((32, 64), 0x7F7F, dtype=np.uint16)
    out = oracle.mxfp8_quantize(m)
    assert np.all(out["sf_row"] == 247) and np.all(out["q_row"] == 0x78)
    assert np.all(out["sf_colT"] == 247) and np.all(out["q_colT"] == 0x78)


def test_rejects_non_finite():
    x = np.zeros((1, 32), dtype=np.uint16)
    x[0, 3] = 0x7F80
    with pytest.raises(ValueError):
        oracle.mxfp8_quantize(x)
