"""Pin the oracle's float64 shortcuts against exact rational arithmetic (no GPU).

The oracle forms NVFP4 quotients in float64 and rounds the result again onto fp32 / E4M3 / E2M1;
its docstring argues this equals one rounding of the real quotient. Here every such decision is
recomputed with Python Fractions (exact), by a different procedure: nearest representable value by
exact distance, ties to the even code. Exhaustive over bf16 where the domain is bf16 alone.
"""
import bisect
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.formats import E2M1_VALUES, E4M3_VALUES

F_E4M3 = [Fraction(float(v)) for v in E4M3_VALUES]
F_E2M1 = [Fraction(float(v)) for v in E2M1_VALUES]


def exact_rne_fp32(a):
    """Nearest fp32 to the non-negative rational a, ties to even (subnormals kept)."""
    if a == 0:
        return 0.0
    E = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** E > a:
        E -= 1
    while Fraction(2) ** (E + 1) <= a:
        E += 1
    qexp = max(E - 23, -149)
    q = a / (Fraction(2) ** qexp)
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return float(n * Fraction(2) ** qexp)


def exact_rne_table(a, table):
    """Code of the entry of ``table`` (exact, increasing) nearest to a >= 0; ties to even code;
    values beyond the last entry saturate."""
    if a >= table[-1]:
        return len(table) - 1
    i = bisect.bisect_right(table, a) - 1
    lo, hi = a - table[i], table[i + 1] - a
    if lo < hi:
        return i
    if hi < lo:
        return i + 1
    return i if i % 2 == 0 else i + 1


def test_token_scale_exhaustive_over_bf16():
    bits = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)
    a = oracle.bf16_bits_to_f64(bits)
    got = oracle.nvfp4_token_scale(a)
    for av, g in zip(a, got):
        assert float(g) == exact_rne_fp32(Fraction(float(av)) / 2688), av


def _bf16_values(rng, n, lo_exp, hi_exp):
    m = rng.integers(128, 256, n)
    e = rng.integers(lo_exp, hi_exp, n)
    return np.ldexp(m.astype(np.float64), e - 7)


def _check_rows(x, s):
    """Quantize rows with the oracle and recheck every scale and code exactly."""
    q, sf = oracle.nvfp4_quantize_rows(x, s)
    codes = oracle.unpack_e2m1(q)
    R, C = x.shape
    for r in range(R):
        fs = Fraction(float(np.float32(s[r])))
        for b in range(C // 16):
            blk = x[r, 16 * b:16 * b + 16]
            amax = Fraction(float(np.abs(blk).max()))
            want_sf = 0 if fs == 0 else exact_rne_table(amax / (6 * fs), F_E4M3)
            assert sf[r, b] == want_sf, (r, b)
            d = F_E4M3[want_sf] * fs
            for j in range(16):
                xv = float(blk[j])
                mag = 0 if d == 0 else exact_rne_table(abs(Fraction(xv)) / d, F_E2M1)
                want = mag | (8 if np.signbit(xv) else 0)
                assert codes[r, 16 * b + j] == want, (r, b, j, xv)


def test_scales_and_codes_random_exact():
    rng = np.random.default_rng(11)
    R = 300
    x = np.empty((R, 64))
    for r in range(R):
        x[r] = _bf16_values(rng, 64, -20, 20) * rng.choice([-1, 1], 64)
        x[r, rng.integers(0, 64, 8)] *= 2.0 ** -rng.integers(0, 30, 8)   # small blocks / sub-scales
    amax = np.abs(x).max(axis=1)
    _check_rows(x, oracle.nvfp4_token_scale(amax))


def test_scales_and_codes_at_exact_ties():
    # s = 2^k exactly (token amax = 42 * 2^(k+6)); blocks built from E4M3 and E2M1 midpoints so
    # that both roundings meet exact ties, plus the neighbouring bf16 values on each side.
    rng = np.random.default_rng(12)
    rows = []
    scales = []
    mids4 = [(F_E4M3[i] + F_E4M3[i + 1]) / 2 for i in range(len(F_E4M3) - 1)]
    mids2 = [(F_E2M1[i] + F_E2M1[i + 1]) / 2 for i in range(7)]
    tries = 0
    while len(rows) < 400 and tries < 100000:
        tries += 1
        k = int(rng.integers(-40, 20))
        s = Fraction(2) ** k
        m = mids4[int(rng.integers(20, len(mids4)))]
        amax_b = 6 * m * s
        f32 = np.float32(float(amax_b))
        if Fraction(float(f32)) != amax_b or (int(f32.view(np.uint32)) & 0xFFFF):
            continue                                    # not exactly a bf16 value
        sfc = exact_rne_table(amax_b / (6 * s), F_E4M3)
        d = F_E4M3[sfc] * s
        blk = [float(amax_b)]
        for _ in range(15):
            t = mids2[int(rng.integers(0, 7))] * d
            v = float(t)
            bv = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits_rne(np.array([v])))[0]
            step = 2.0 ** (np.frexp(bv)[1] - 8) if bv else 0.0
            blk.append(float(rng.choice([bv, bv + step, bv - step])) * float(rng.choice([-1, 1])))
        row = np.array(blk)
        row = np.minimum(np.abs(row), float(amax_b)) * np.sign(row)
        token = np.concatenate([row, [42.0 * float(s) * 64.0], np.zeros(15)])
        rows.append(token)
        scales.append(float(s))
    x = np.array(rows)
    s = oracle.nvfp4_token_scale(np.abs(x).max(axis=1))
    assert np.array_equal(s.astype(np.float64), np.array(scales))
    _check_rows(x, s)


@pytest.mark.parametrize("k", [-125, -126, -127, -140, -149])
def test_subnormal_token_scales_exact(k):
    # tiny tokens: s_tok subnormal in fp32; the float64 path must still decide exactly
    rng = np.random.default_rng(13 + (-k))
    amax = 2688.0 * 2.0 ** k * 1.3
    x = _bf16_values(rng, 64, -10, 0).reshape(1, 64) * 2.0 ** (k + 11)
    x[0, 0] = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits_rne(np.array([amax])))[0]
    x = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits_rne(x))
    s = oracle.nvfp4_token_scale(np.abs(x).max(axis=1))
    _check_rows(x, s)
