"""The NVFP4 quantizers' product path, checked on the CPU against the oracle's exact codes.

A scope (one token row, or one expert matrix) with coarse scale s may encode its elements as
E2M1_RNE_satfinite(RN_fp32(x * g)) for a per-class multiplier g near 1 / (v s) (v the block
scale's E4M3 value), instead of comparing each element with the block's exact boundaries. The
kernels allow this only when, for every E4M3 mantissa class (codes 8 + f), one of five candidate
multipliers (RN(1 / RN(v s)) and its neighbours 1 and 2 ulps away) gives the two bf16 neighbours
of each of the seven E2M1 boundaries the right code; monotonicity of both roundings then makes
every bf16 element right, and a block with code 8 (d + 1) + f (or a subnormal code) uses g 2^-d.

These tests restate that check in numpy (as the kernels state it), then compare the product codes
of every bf16 value around the thresholds with the oracle's exact codes, for the classes that
pass, at several exponent steps, for generic scopes and for scopes of bf16 maxima (whose
RN(amax / 2688) puts bf16 values close to boundaries). They also show that the power-of-two scopes
of the GPU parity inputs fail the check for some class (so those rows exercise the boundary
comparison) while nearly all other scopes pass it.
"""
import numpy as np
import pytest

import oracle

F32 = np.float32


def _bf16_window(lo, hi):
    """All positive bf16 values in [lo, hi] (float64 bounds), as float64, ascending."""
    b0 = int(np.array(lo, dtype=F32).view(np.uint32)) >> 16
    b1 = (int(np.array(hi, dtype=F32).view(np.uint32)) >> 16) + 1
    bits = np.arange(max(b0, 1), min(b1, 0x7F80), dtype=np.uint32)
    return (bits << 16).view(F32).astype(np.float64), bits


def _exact_mag(x, v, s):
    # the oracle's decision: E2M1 RNE of x / (v s), magnitude code
    return oracle.round_to_e2m1(x / (v * float(s))) & 7


def _prod_mag(x, g):
    y = (x.astype(F32) * F32(g)).astype(F32)            # one fp32 rounding, as __fmul_rn
    return oracle.round_to_e2m1(y.astype(np.float64)) & 7


def _class_g0(v, s):
    g = F32(1.0) / (F32(v) * F32(s))                    # RN(1 / RN(v s)), as __frcp_rn(__fmul_rn)
    e = (int(np.array(g, dtype=F32).view(np.uint32)) >> 23) & 0xFF
    return g if 16 <= e <= 250 else F32(0.0)


CANDIDATE_ULPS = (0, -1, 1, -2, 2)                      # tried in this order


def _candidate(g0, c):
    return np.array(int(np.array(g0, dtype=F32).view(np.uint32)) + CANDIDATE_ULPS[c], dtype=np.uint32).view(F32)


def _class_multiplier(f, s):
    """The kernels' check for class f (E4M3 code 8 + f) of a scope with coarse scale s: the first
    candidate multiplier that passes at every boundary, or None."""
    v = (8 + f) * 2.0 ** -9
    g0 = _class_g0(v, s)
    if g0 == 0:
        return None
    x, bits = _bf16_window(v * float(s) * 2.0 ** -4, v * float(s) * 2.0 ** 4)
    ex = _exact_mag(x, v, s)
    pairs = []
    for j in range(7):
        i = int(np.argmax(ex > j))                       # b_j: smallest bf16 with code > j
        assert ex[i] > j and i > 0
        pairs.append((j, x[i], x[i - 1]))                # consecutive bf16 values
    for c in range(len(CANDIDATE_ULPS)):
        g = _candidate(g0, c)
        if all(_prod_mag(np.array([b]), g)[0] > j and _prod_mag(np.array([below]), g)[0] <= j
               for j, b, below in pairs):
            return g
    return None


def _class_passes(f, s):
    return _class_multiplier(f, s) is not None


def _scope_passes(s):
    return all(_class_passes(f, s) for f in range(8))


def _code_value(c):
    return float(oracle.e4m3_decode(np.array([c], dtype=np.uint8))[0])


def _code_class_step(c):
    # code 8 (d + 1) + f -> (f, d); subnormal code c = (8 + f') 2^(p - 3) -> (f', p - 3)
    if c >= 8:
        return c & 7, (c >> 3) - 1
    p = c.bit_length() - 1
    return (c << (3 - p)) - 8, p - 3


def _random_scopes(n, seed):
    rng = np.random.default_rng(seed)
    return (np.exp2(rng.uniform(-85, 110, n)) * rng.uniform(1, 2, n)).astype(F32)


def _amax_scopes(n, seed):
    # s = RN_fp32(amax / 2688) for bf16 maxima, as the quantizers compute it
    rng = np.random.default_rng(seed)
    a = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits_rne(np.exp(rng.uniform(-60, 60, n))))
    return oracle.nvfp4_token_scale(a)


@pytest.mark.parametrize("kind,seed", [("random", 0), ("random", 1), ("amax", 2), ("amax", 3)])
def test_product_codes_equal_exact_codes_where_the_check_passes(kind, seed):
    checked = 0
    scopes = _random_scopes(6, seed) if kind == "random" else _amax_scopes(6, seed)
    for s in scopes:
        for f in range(8):
            if not _class_passes(f, s):
                continue
            g = _class_multiplier(f, s)
            # every code of this class: subnormal codes, and normal codes at several exponent steps
            codes = [c for c in range(1, 0x7F) if _code_class_step(c)[0] == f]
            for c in codes[:2] + codes[len(codes) // 2:len(codes) // 2 + 1] + codes[-2:]:
                v = _code_value(c)
                d = _code_class_step(c)[1]
                assert np.isclose(v, (8 + f) * 2.0 ** -9 * 2.0 ** d, rtol=0, atol=0)
                g_c = F32(g * F32(2.0 ** -d))
                x, _ = _bf16_window(v * float(s) * 2.0 ** -4, min(v * float(s) * 2.0 ** 4, 3.3e38))
                if x.size == 0:
                    continue
                got = _prod_mag(x, g_c)
                want = _exact_mag(x, v, s)
                assert np.array_equal(got, want), (float(s), f, c)
                checked += 1
    assert checked > 20


def test_power_of_two_scopes_take_the_boundary_comparison():
    # the GPU parity inputs' "nice" rows have s = 2^k, k in [-10, 10): each must fail the check for
    # some class, so that the boundary comparison stays covered by those tests
    for k in range(-10, 10):
        assert not _scope_passes(F32(2.0 ** k)), k


def test_generic_scopes_take_the_product_path():
    s = _random_scopes(40, 7)
    passed = sum(_scope_passes(x) for x in s)
    assert passed >= 38, passed
    s = _amax_scopes(100, 8)
    passed = sum(_scope_passes(x) for x in s)
    assert passed >= 90, passed


def test_one_candidate_would_not_do():
    # with RN(1 / RN(v s)) alone, scopes of bf16 maxima fail about half of the time: the check's
    # candidates are what make the product path the common case
    s = _amax_scopes(100, 8)
    alone = 0
    for x in s:
        ok = True
        for f in range(8):
            v = (8 + f) * 2.0 ** -9
            g0 = _class_g0(v, x)
            xs, _ = _bf16_window(v * float(x) * 2.0 ** -4, v * float(x) * 2.0 ** 4)
            if g0 == 0 or not np.array_equal(_prod_mag(xs, g0), _exact_mag(xs, v, x)):
                ok = False
                break
        alone += ok
    assert alone <= 70, alone


def test_the_check_catches_a_wrong_multiplier():
    # a multiplier one ulp off on a scope with ties on the boundaries is rejected for some class
    s = F32(1.0)
    bad = 0
    for f in range(8):
        v = (8 + f) * 2.0 ** -9
        g = _class_g0(v, s)
        g_off = np.nextafter(g, F32(np.inf), dtype=F32)
        x, _ = _bf16_window(v * 2.0 ** -4, v * 2.0 ** 4)
        ex = _exact_mag(x, v, s)
        if not np.array_equal(_prod_mag(x, g_off), ex):
            bad += 1
    assert bad > 0


def _class_pairs(f, s):
    v = (8 + f) * 2.0 ** -9
    x, _ = _bf16_window(v * float(s) * 2.0 ** -4, v * float(s) * 2.0 ** 4)
    ex = _exact_mag(x, v, s)
    pairs = []
    for j in range(7):
        i = int(np.argmax(ex > j))
        pairs.append((j, x[i], x[i - 1]))
    return pairs


def _miss(pairs, g):
    # bit 0: some boundary's product keeps its code at or below the threshold (g too small);
    # bit 1: some value just below a boundary gets a code above it (g too large)
    m = 0
    for j, b, below in pairs:
        if _prod_mag(np.array([b]), g)[0] <= j:
            m |= 1
        if _prod_mag(np.array([below]), g)[0] > j:
            m |= 2
    return m


def _directed_multiplier(f, s):
    """The kernels' search as they run it: candidate 0, then up to two steps (1 and 2 ulps) towards
    the side it missed on, stopping at the first pass or at a miss on the other side."""
    v = (8 + f) * 2.0 ** -9
    g0 = _class_g0(v, s)
    if g0 == 0:
        return None
    pairs = _class_pairs(f, s)
    m0 = _miss(pairs, g0)
    if m0 == 0:
        return g0
    if m0 == 3:
        return None
    step = 1 if m0 == 1 else -1
    for k in (1, 2):
        g = np.array(int(np.array(g0, dtype=F32).view(np.uint32)) + k * step, dtype=np.uint32).view(F32)
        mk = _miss(pairs, g)
        if mk == 0:
            return g
        if mk != m0:
            return None
    return None


@pytest.mark.parametrize("kind,seed", [("random", 11), ("amax", 12), ("amax", 13)])
def test_directed_search_picks_the_first_passing_candidate(kind, seed):
    # the candidates that pass form one run around RN(1 / RN(v s)) (both codes are monotone in g),
    # so stepping away from the side candidate 0 misses on finds what the order 0, -1, +1, -2, +2 finds
    scopes = _random_scopes(12, seed) if kind == "random" else _amax_scopes(24, seed)
    moved = 0
    for s in scopes:
        for f in range(8):
            want = _class_multiplier(f, s)
            got = _directed_multiplier(f, s)
            assert (want is None) == (got is None), (float(s), f)
            if want is not None:
                assert F32(want) == F32(got), (float(s), f)
                moved += F32(want) != _class_g0((8 + f) * 2.0 ** -9, s)
            # the passing candidates are consecutive
            g0 = _class_g0((8 + f) * 2.0 ** -9, s)
            if g0 != 0:
                pairs = _class_pairs(f, s)
                ok = [_miss(pairs, _candidate(g0, c)) == 0 for c in (3, 1, 0, 2, 4)]   # -2 .. +2
                runs = sum(1 for i in range(5) if ok[i] and (i == 0 or not ok[i - 1]))
                assert runs <= 1, (float(s), f, ok)
    if kind == "amax":
        assert moved > 0                     # scopes of bf16 maxima do need the steps
