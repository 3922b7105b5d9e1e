"""Element and scale formats of MXFP8 and NVFP4, written from their definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages name the formats but do not spell out their bit layouts:
  * MXFP8: 32 consecutive E4M3 values share one E8M0 power-of-two scale [Miles-zh, section
    "为什么需要 Blackwell 原生方案？", MXFP8 paragraph; Miles-vi, "Bối cảnh định dạng / MXFP8"].
  * NVFP4: E2M1 values, one E4M3 scale per 16 values, plus a coarse FP32 scale [Miles-zh, same
    section, NVFP4 paragraph; Miles-vi, "Bối cảnh định dạng / NVFP4"; NVFP4-ru, second paragraph].
The plainest reading is the OCP microscaling definitions, which the bit layouts below follow:
  E4M3 ("E4M3FN"): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
                   S.1111.111 is NaN, largest finite value 448.
  E2M1:            1 sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
                   {0, 0.5, 1, 1.5, 2, 3, 4, 6} (the value set is fixed by the method statement).
  E8M0:            unsigned byte b encodes 2^(b-127); 0xFF is NaN.
  BF16:            1 sign, 8 exponent bits (bias 127), 7 mantissa bits.
"""

import numpy as np


# ----------------------------------------------------------------------------------------------
# Decoding tables, built from the bit-field definitions above.
# ----------------------------------------------------------------------------------------------

def _decode_e4m3(code):
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:  # subnormal: 2^(1-7) * man/8
        return sign * man * 2.0 ** -9
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


def _decode_e2m1(code):
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:  # subnormal: 2^(1-1) * man/2
        return sign * man * 0.5
    return sign * (1.0 + man / 2.0) * 2.0 ** (exp - 1)


#: value of every E4M3 code 0..255 (NaN for 0x7F / 0xFF)
E4M3_TABLE = np.array([_decode_e4m3(c) for c in range(256)], dtype=np.float64)
#: value of every E2M1 code 0..15
E2M1_TABLE = np.array([_decode_e2m1(c) for c in range(16)], dtype=np.float64)

#: non-negative finite E4M3 values in code order (codes 0x00..0x7E are increasing in value)
E4M3_VALUES = E4M3_TABLE[:0x7F].copy()
#: non-negative E2M1 values in code order (codes 0..7)
E2M1_VALUES = E2M1_TABLE[:8].copy()
E4M3_MAX = float(E4M3_VALUES[-1])   # 448
E2M1_MAX = float(E2M1_VALUES[-1])   # 6


def e4m3_decode(codes):
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e2m1_decode(codes):
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def e8m0_decode(codes):
    """2^(b-127) for every byte b (0xFF -> NaN)."""
    b = np.asarray(codes, dtype=np.int64)
    out = np.ldexp(1.0, b - 127)
    return np.where(b == 0xFF, np.nan, out)


# ----------------------------------------------------------------------------------------------
# BF16 <-> float64
# ----------------------------------------------------------------------------------------------

def bf16_bits_to_f64(bits):
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits_rne(v):
    """Round float64 values to bf16 once, to nearest with ties to even; returns uint16 bits.

    Written from the definition: the bf16 quantum at |v| is 2^(floor(log2|v|) - 7) in the normal
    range and 2^-133 below 2^-126; |v| / quantum is an exact power-of-two scaling, np.rint rounds
    it to the nearest integer with ties to even, and results of 2^128 or more overflow to infinity.
    """
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v) | np.isinf(v)):
        raise ValueError("NaN input")
    a = np.abs(v)
    _, E = np.frexp(a)                      # a = f * 2^E, f in [0.5, 1)  ->  floor(log2 a) = E - 1
    q_exp = np.where(a >= 2.0 ** -126, (E - 1) - 7, -133)
    r = np.ldexp(np.rint(np.ldexp(a, -q_exp)), q_exp)
    r = np.where(np.isinf(a), np.inf, r)
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    sign = np.signbit(v).astype(np.uint16) << 15
    return bits | sign


# ----------------------------------------------------------------------------------------------
# Round-to-nearest-even onto a value table (satfinite)
# ----------------------------------------------------------------------------------------------

def _round_to_table(v, values, sign_bit):
    """Round each real v once to the nearest entry of ``values`` (ties to the even code).

    ``values`` are the non-negative finite values of the format in code order, so the code of a
    magnitude equals its index. Magnitudes above the largest value saturate to it (satfinite).
    The sign is carried separately, so -0.0 and negative values that round to zero keep the sign
    bit, as an IEEE conversion does. Comparisons are against exact midpoints, so the rounding is
    decided exactly for every float64 input.
    """
    v = np.asarray(v, dtype=np.float64)
    if np.any(np.isnan(v)):
        raise ValueError("NaN input to rounding")
    a = np.abs(v)
    n = len(values)
    i = np.searchsorted(values, a, side="right") - 1          # values[i] <= a < values[i+1]
    i = np.clip(i, 0, n - 1)
    nxt = np.minimum(i + 1, n - 1)
    mid = (values[i] + values[nxt]) * 0.5                      # exact: few significant bits
    go_up = (i < n - 1) & ((a > mid) | ((a == mid) & (i % 2 == 1)))
    code = i + go_up.astype(np.int64)
    sign = np.signbit(v).astype(np.int64) * sign_bit
    return (code | sign).astype(np.uint8)


def round_to_e4m3(v):
    """E4M3 code of RNE_satfinite(v) for real (float64) v."""
    return _round_to_table(v, E4M3_VALUES, 0x80)


def round_to_e2m1(v):
    """E2M1 code (0..15) of RNE_satfinite(v) for real (float64) v."""
    return _round_to_table(v, E2M1_VALUES, 0x8)


# ----------------------------------------------------------------------------------------------
# E8M0 scale exponent
# ----------------------------------------------------------------------------------------------

def e8m0_exponent(amax):
    """Smallest integer e with amax <= 448 * 2^e, clamped to the E8M0 range [-127, 127].

    [Miles-zh, "为什么需要 Blackwell 原生方案？": because E8M0 scales are powers of two, the
    decoded scale is rounded up so the block maximum is not clipped; Miles-vi, "Bối cảnh định
    dạng / MXFP8", same statement.] Reading: "rounded up" = the smallest power of two that keeps
    amax <= 448 (the largest E4M3 value) after scaling; amax = 0 gives the lowest scale, -127.
    """
    a = np.asarray(amax, dtype=np.float64)
    if np.any(~np.isfinite(a)) or np.any(a < 0):
        raise ValueError("amax must be finite and non-negative")
    safe = np.where(a > 0, a, 1.0)
    _, E = np.frexp(safe)                   # safe < 2^E
    e = E.astype(np.int64) - 9              # 448 * 2^(E-9) = 0.875 * 2^E: within a factor 2
    for _ in range(3):                      # exact adjustment to the smallest valid e
        e = np.where(safe > np.ldexp(448.0, e), e + 1, e)
    for _ in range(3):
        e = np.where(safe <= np.ldexp(448.0, e - 1), e - 1, e)
    e = np.where(a > 0, e, -127)
    return np.clip(e, -127, 127)
