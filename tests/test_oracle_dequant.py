"""Pins for the oracle's BF16 dequantization (no GPU): exactness closed form, torch's float8
decode as an independent route, and quantize -> dequantize error bounds."""
import numpy as np
import torch

import oracle


def _bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_mxfp8_dequant_via_torch_float8():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((64, 128)) * np.exp(rng.uniform(-10, 10, (64, 1)))
    out = oracle.mxfp8_quantize(_bits(x), colwise=False)
    q, sf = out["q_row"], out["sf_row"]
    ours = oracle.dequantize_mxfp8(q, sf)
    # independent route: torch decodes E4M3, times 2^(sf-127) in fp32 (exact here), cast to bf16
    v = torch.from_numpy(q).view(torch.float8_e4m3fn).float()
    scale = torch.pow(2.0, torch.from_numpy(sf.astype(np.float32) - 127)).repeat_interleave(32, 1)
    ref = (v * scale).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_mxfp8_quantize_dequantize_error_bound():
    rng = np.random.default_rng(1)
    x = oracle.bf16_bits_to_f64(_bits(rng.standard_normal((32, 256)) * 10))
    out = oracle.mxfp8_quantize(oracle.f64_to_bf16_bits_rne(x), colwise=False)
    y = oracle.bf16_bits_to_f64(oracle.dequantize_mxfp8(out["q_row"], out["sf_row"]))
    amax = np.abs(x).reshape(32, 8, 32).max(axis=2).repeat(32, axis=1)
    # E4M3 keeps 4 significant bits on normals (half-ulp 2^-4) and a 2^-9 * 2^e floor below
    e = np.ldexp(1.0, oracle.e8m0_exponent(amax))
    assert np.all(np.abs(y - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * e) * (1 + 2 ** -7) + 1e-300)


def test_nvfp4_dequant_closed_form():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((16, 64)) * np.exp(rng.uniform(-6, 6, (16, 1)))
    q, sf, s = oracle.nvfp4_quantize_per_token(_bits(x))
    y = oracle.bf16_bits_to_f64(oracle.dequantize_nvfp4(q, sf, s))
    codes = oracle.unpack_e2m1(q)
    vals = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])[codes]
    exact = vals * oracle.e4m3_decode(sf).repeat(16, axis=1) * s.astype(np.float64)[:, None]
    # exact product rounds once to bf16 (8 significant bits): relative error <= 2^-8
    nz = exact != 0
    assert np.all(np.abs(y[nz] - exact[nz]) <= np.abs(exact[nz]) * 2.0 ** -8)
    assert np.all(y[~nz] == 0)
    # and when the product is itself a bf16 value, it comes back unchanged
    bf = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits_rne(exact))
    same = bf == exact
    assert np.all(y[same] == exact[same])


def test_nvfp4_quantize_dequantize_error_bound():
    rng = np.random.default_rng(3)
    x = oracle.bf16_bits_to_f64(_bits(rng.standard_normal((64, 128))))
    q, sf, s = oracle.nvfp4_quantize_per_token(oracle.f64_to_bf16_bits_rne(x))
    y = oracle.bf16_bits_to_f64(oracle.dequantize_nvfp4(q, sf, s))
    d = (oracle.e4m3_decode(sf) * s.astype(np.float64)[:, None]).repeat(16, axis=1)
    # E2M1 step is at most 2 * d (between 4 and 6): error <= d away from saturation, plus bf16 rounding
    assert np.all(np.abs(y - x) <= d * 1.0 + np.abs(y) * 2.0 ** -8 + np.abs(x) * 2.0 ** -4)
