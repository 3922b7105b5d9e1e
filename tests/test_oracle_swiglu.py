"""Pins of the SwiGLU oracle (oracle/swiglu.py) against math.exp, float64 silu and closed forms.

The exp is our own float32 algorithm (Cody-Waite reduction + Taylor polynomial); these tests fix
it against the real function, so a dropped term, a wrong constant or a wrong reduction step fails.
The SwiGLU is checked against float64 silu(g) * u for every bf16 gate from -bf16 max to 100,
including the gates where exp(-g) leaves float32's range, with large and small up values.
"""
import math

import numpy as np

import oracle
from oracle import swiglu

BF16_MAX = 3.3895313892515355e38


def _ulp32(v):
    """float32 ulp of |v| with an unbounded exponent (a 24-bit significand at any scale)."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(v, 1e-300)))
    return 2.0 ** (e - 23)


def test_exp_parts_within_four_float32_ulp():
    # measured worst case 2.94 ulp (float32 Horner rounding); a dropped Taylor term alone costs
    # 20-40 ulp at |r| = ln2/2, a wrong reduction constant far more
    x = np.concatenate([np.linspace(-87.0, 300.0, 400001), np.arange(-87, 301, dtype=np.float64),
                        [0.0, -0.0, 1e-30, -1e-30, 0.5 * math.log(2), -0.5 * math.log(2),
                         88.72283935546875, 88.7228317260742]]).astype(np.float32)
    p, n = swiglu.exp_parts(x)
    got = np.ldexp(p.astype(np.float64), n.astype(np.int32))
    ref = np.exp(x.astype(np.float64))
    assert (np.abs(got - ref) <= 4 * _ulp32(ref)).all()
    p0, n0 = swiglu.exp_parts(np.float32(0.0))
    assert p0 == np.float32(1.0) and n0 == 0


def test_exp_f32_normal_range():
    x = np.linspace(-87.0, 87.0, 100001).astype(np.float32)
    got = swiglu.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    assert (np.abs(got - ref) <= 4 * _ulp32(ref)).all()
    assert swiglu.exp_f32(np.float32(-200.0)) == swiglu.exp_f32(np.float32(-87.0))


def _bits(v):
    return oracle.f64_to_bf16_bits_rne(np.asarray(v, dtype=np.float64))


def _silu_times_u(gf, uf):
    with np.errstate(over="ignore"):
        return gf * uf / (1.0 + np.exp(-gf))


def _check_against_float64(g_bits, u_bits):
    h = oracle.bf16_bits_to_f64(swiglu.swiglu_bf16_bits(g_bits, u_bits))
    ref = _silu_times_u(oracle.bf16_bits_to_f64(g_bits), oracle.bf16_bits_to_f64(u_bits))
    inside = np.abs(ref) < BF16_MAX            # results that overflow are outside the contract
    # one bf16 rounding (2^-8 relative; 2^-134 absolute among subnormals) plus the float32 steps
    bound = np.abs(ref) * (2.0 ** -8 + 2.0 ** -20) + 2.0 ** -134 + 2.0 ** -149
    bad = inside & ~(np.abs(h - ref) <= bound)
    assert not bad.any(), (g_bits[bad][:5], u_bits[bad][:5] if np.ndim(u_bits) else u_bits)
    # the sign of a zero result is the sign of g * u
    zero = inside & (h == 0)
    sg = np.signbit(oracle.bf16_bits_to_f64(g_bits)) ^ np.signbit(oracle.bf16_bits_to_f64(u_bits))
    assert np.array_equal(np.signbit(h)[zero], np.broadcast_to(sg, h.shape)[zero])
    return inside.sum()


def test_swiglu_every_bf16_gate_against_float64():
    # every finite bf16 gate from -bf16 max up to 100 (about 33 000 values), against up values from
    # bf16 max down to the smallest subnormal: covers exp(-g) inside float32's range, beyond it
    # (g < -88.7: the unbounded-exponent form) and beyond the clamp at 300
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    gv = oracle.bf16_bits_to_f64(allb)
    g_bits = allb[np.isfinite(gv) & (gv <= 100.0)]
    for u in [1.0, -1.0, 1e30, -1e30, 3.3e38, -3.3e38, 7.0, 1e-30, 2.0 ** -133, -0.0]:
        n = _check_against_float64(g_bits, np.full(g_bits.shape, _bits(u), dtype=np.uint16))
        assert n > 30000


def test_swiglu_random_pairs_against_float64():
    rng = np.random.default_rng(0)
    g = _bits(rng.standard_normal(200000) * np.exp(rng.uniform(-4, 6, 200000)))
    u = _bits(rng.standard_normal(200000) * np.exp(rng.uniform(-90, 88, 200000)))
    _check_against_float64(g, u)
    # the gate is the first operand: swapping the operands changes the result
    assert not np.array_equal(swiglu.swiglu_bf16_bits(u, g), swiglu.swiglu_bf16_bits(g, u))


def test_swiglu_special_cases():
    def h(g, u):
        return int(swiglu.swiglu_bf16_bits(_bits(g), _bits(u)))
    # silu(0) = 0 with the sign of g times u
    assert h(0.0, 3.0) == 0x0000
    assert h(-0.0, 3.0) == 0x8000
    # large positive gate: exp(-g) vanishes, d = 1 exactly, so h = RN_bf16(g u)
    for g, u in [(100.0, 1.5), (1e10, -2.0), (90.0, 0.25)]:
        assert h(g, u) == int(_bits(np.float32(g) * np.float32(u)))
    # large negative gate, exp(-g) beyond float32's range: silu(g) u is still g e^g u
    g, u = oracle.bf16_bits_to_f64(_bits(-90.0)), oracle.bf16_bits_to_f64(_bits(1e30))
    ref = g * u / (1.0 + math.exp(-g))                       # -7.38e-8
    assert h(-90.0, 1e30) == int(_bits(ref)) and abs(ref + 7.38e-8) < 1e-10
    # ... and rounds to a signed zero once it is below half the smallest bf16 subnormal
    assert h(-100.0, 1.0) == 0x8000                          # -3.7e-42
    assert h(-3e38, 1.0) == 0x8000
    assert h(-3e38, -1.0) == 0x0000
    assert h(-3e38, 3e38) == 0x8000                          # clamped exp: still a zero
    assert h(-1e5, -3.3e38) == 0x0000
    # silu(1) * 1 = 1 / (1 + e^-1)
    assert h(1.0, 1.0) == int(_bits(1.0 / (1.0 + math.exp(-1.0))))


def test_swiglu_two_forms_agree_on_their_overlap():
    # for 87 < -g < 88.3 (n <= 127) both the IEEE float32 steps and the unbounded-exponent form are defined;
    # the oracle takes the latter there, and it must give what the plain float32 steps give
    g32 = -np.linspace(87.0001, 88.3, 5000).astype(np.float32)
    u32 = np.float32(3.0e38) * np.linspace(-1.0, 1.0, 5000).astype(np.float32)
    p, n = swiglu.exp_parts((-g32).astype(np.float32))
    assert (n <= 127).all()
    two_n = np.ldexp(np.float32(1.0), n.astype(np.int32)).astype(np.float32)   # normal up to 2^127
    e = (p * two_n).astype(np.float32)
    d = (np.float32(1.0) + e).astype(np.float32)
    plain = ((g32 / d).astype(np.float32) * u32).astype(np.float32)
    assert np.isfinite(d).all()
    assert np.array_equal(swiglu.swiglu_f32(g32, u32).view(np.uint32), plain.view(np.uint32))


def test_swiglu_rows_splits_gate_then_up():
    rng = np.random.default_rng(1)
    gu = _bits(rng.standard_normal((5, 64)))
    h = swiglu.swiglu_rows(gu)
    assert h.shape == (5, 32)
    assert np.array_equal(h, swiglu.swiglu_bf16_bits(gu[:, :32], gu[:, 32:]))
