"""Pins of the SwiGLU oracle (oracle/swiglu.py) against math.exp, float64 silu and closed forms.

The exp is our own float32 algorithm (Cody-Waite reduction + Taylor polynomial); these tests fix
it against the real function, so a dropped term, a wrong constant or a wrong reduction step fails.
"""
import math

import numpy as np

import oracle
from oracle import swiglu


def _ulp32(v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return 2.0 ** (e - 23)


def test_exp_within_four_float32_ulp():
    # measured worst case 2.9 ulp (float32 Horner rounding); a dropped Taylor term alone costs
    # 20-40 ulp at |r| = ln2/2, a wrong reduction constant far more
    x = np.concatenate([np.linspace(-87.0, 88.0, 200001), np.arange(-87, 89, dtype=np.float64),
                        [0.0, -0.0, 1e-30, -1e-30, 0.5 * math.log(2), -0.5 * math.log(2)]]).astype(np.float32)
    got = swiglu.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    assert (np.abs(got - ref) <= 4 * _ulp32(ref)).all()
    assert swiglu.exp_f32(np.float32(0.0)) == np.float32(1.0)


def test_exp_clamps_outside_the_normal_range():
    assert swiglu.exp_f32(np.float32(-200.0)) == swiglu.exp_f32(np.float32(-87.0))
    assert swiglu.exp_f32(np.float32(500.0)) == swiglu.exp_f32(np.float32(88.0))
    assert np.isfinite(swiglu.exp_f32(np.float32(88.0)))


def _bits(v):
    return oracle.f64_to_bf16_bits_rne(np.asarray(v, dtype=np.float64))


def test_swiglu_matches_float64_within_one_bf16_rounding():
    rng = np.random.default_rng(0)
    g = _bits(rng.standard_normal(200000) * np.exp(rng.uniform(-4, 3, 200000)))
    u = _bits(rng.standard_normal(200000) * np.exp(rng.uniform(-4, 3, 200000)))
    h = oracle.bf16_bits_to_f64(swiglu.swiglu_bf16_bits(g, u))
    gf, uf = oracle.bf16_bits_to_f64(g), oracle.bf16_bits_to_f64(u)
    ref = gf / (1.0 + np.exp(-gf)) * uf
    # one bf16 rounding (2^-8 relative) plus the float32 steps (a few 2^-24)
    assert (np.abs(h - ref) <= np.abs(ref) * (2.0 ** -8 + 2.0 ** -20) + 1e-37).all()
    # the gate is the first operand: swapping the operands changes the result
    assert not np.array_equal(swiglu.swiglu_bf16_bits(u, g), swiglu.swiglu_bf16_bits(g, u))


def test_swiglu_special_cases():
    # silu(0) = 0 with the sign of g times u
    assert int(swiglu.swiglu_bf16_bits(_bits(0.0), _bits(3.0))) == 0x0000
    assert int(swiglu.swiglu_bf16_bits(_bits(-0.0), _bits(3.0))) == 0x8000
    # large positive gate: silu(g) = g to float32 precision, so h = RN_bf16(g u)
    for g, u in [(100.0, 1.5), (1e10, -2.0), (90.0, 0.25)]:
        assert int(swiglu.swiglu_bf16_bits(_bits(g), _bits(u))) == int(_bits(np.float32(g) * np.float32(u)))
    # large negative gate: silu(g) is tiny (here of the clamped exp), with the sign of g * u
    h = oracle.bf16_bits_to_f64(swiglu.swiglu_bf16_bits(_bits([-100.0, -1e20]), _bits([2.0, -3.0])))
    assert abs(h[0]) < 1e-30 and h[0] <= 0 and abs(h[1]) < 1e-10 and h[1] >= 0
    # silu(1) * 1 = 1 / (1 + e^-1)
    assert int(swiglu.swiglu_bf16_bits(_bits(1.0), _bits(1.0))) == int(_bits(1.0 / (1.0 + math.exp(-1.0))))


def test_swiglu_rows_splits_gate_then_up():
    rng = np.random.default_rng(1)
    gu = _bits(rng.standard_normal((5, 64)))
    h = swiglu.swiglu_rows(gu)
    assert h.shape == (5, 32)
    assert np.array_equal(h, swiglu.swiglu_bf16_bits(gu[:, :32], gu[:, 32:]))
