"""MXFP8 and per-token NVFP4 quantization and BF16 dequantization, written from the pages.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Inputs are bf16 bit patterns (uint16 numpy arrays, row-major). Outputs are byte arrays in the
canonical layouts: codes [rows, cols] (MXFP8) or packed [rows, cols/2] (NVFP4, element 2j in the
low nibble and 2j+1 in the high nibble), scales [rows, cols/block] row-major. Rearranging scales
into the tensor-core tile layout is ``oracle.layout``.

Exactness: every quotient below is formed in float64 from operands that float64 holds exactly
(bf16 values, fp32 scales, products of at most 31 significant bits) and is then rounded once more
onto a table of at most 5-significant-bit midpoints (or onto fp32 for the token scale). A quotient
a/b with a of at most 8 significant bits and b of at most 28 differs from any such midpoint m
either not at all or by at least 2^-33 relative (a - m*b is a nonzero multiple of the smaller of
the two operands' last-bit weights), while float64 division errs by at most 2^-53 relative. So
the float64 quotient falls on the same side of every midpoint as the real quotient, and ties are
ties exactly when the real quotient is a tie: the two-step rounding equals a single rounding of
the real value. The same argument (midpoints of at most 25 bits against a 5-bit divisor 21 * 2^7)
covers the fp32 token scale. tests/test_oracle_exact.py checks these claims by exact rational
brute force, exhaustively over bf16 where the domain allows.
"""

import numpy as np

from .formats import (
    E2M1_MAX, E4M3_MAX, bf16_bits_to_f64, e2m1_decode, e4m3_decode, e8m0_exponent,
    f64_to_bf16_bits_rne, round_to_e2m1, round_to_e4m3,
)

MXFP8_BLOCK = 32
NVFP4_BLOCK = 16
#: E2M1 max (6) times E4M3 max (448): the coarse scale maps a token's amax onto this.
NVFP4_RANGE = E2M1_MAX * E4M3_MAX   # 2688


def _finite_bf16(x_bits):
    x = bf16_bits_to_f64(x_bits)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite bf16 inputs are outside the quantizer contract")
    return x


# ----------------------------------------------------------------------------------------------
# MXFP8
# ----------------------------------------------------------------------------------------------

def mxfp8_quantize_blocks(x):
    """Quantize each row of real matrix x [R, C] in 1x32 blocks along the row.

    Per block [Miles-zh, "为什么需要 Blackwell 原生方案？" (MXFP8: 32 consecutive E4M3 values share a
    local E8M0 scale; the decoded scale is rounded up so the block max is not clipped)]:
      1. amax = max |x| over the block (exact);
      2. e = smallest integer with amax <= 448 * 2^e, clamped to [-127, 127] (``e8m0_exponent``);
         the scale byte is e + 127;
      3. code = E4M3_RNE_satfinite(x * 2^-e), with x * 2^-e exact in float64.
    Returns (codes uint8 [R, C], scale bytes uint8 [R, C/32]).
    """
    x = np.asarray(x, dtype=np.float64)
    R, C = x.shape
    if C % MXFP8_BLOCK:
        raise ValueError("row length must be a multiple of 32")
    blocks = x.reshape(R, C // MXFP8_BLOCK, MXFP8_BLOCK)
    amax = np.abs(blocks).max(axis=2) if C else np.zeros((R, 0))
    e = e8m0_exponent(amax)
    scaled = np.ldexp(blocks, -e[:, :, None])
    codes = round_to_e4m3(scaled).reshape(R, C)
    return codes, (e + 127).astype(np.uint8)


def mxfp8_quantize(x_bits, rowwise=True, colwise=True):
    """MXFP8 rowwise (1x32) and columnwise (32x1) copies of a bf16 matrix X [M, K].

    [Miles-zh, "方案 1：端到端 MXFP8 强化学习": rowwise 1x32 and columnwise 32x1 blocks are
    numerically different and each is quantized independently from the full-precision data, so
    both copies are materialised during quantization; Miles-fr, "Un quantificateur partagé est le
    véritable mécanisme", same statement.] The columnwise copy is the rowwise rule applied to X^T,
    stored as X^T [K, M] so that each stored row runs along the 32x1 block direction.
    Returns dict with q_row [M,K], sf_row [M,K/32], q_colT [K,M], sf_colT [K,M/32] (as requested).
    """
    x = _finite_bf16(x_bits)
    if x.ndim != 2:
        raise ValueError("X must be 2-D")
    out = {}
    if rowwise:
        out["q_row"], out["sf_row"] = mxfp8_quantize_blocks(x)
    if colwise:
        out["q_colT"], out["sf_colT"] = mxfp8_quantize_blocks(x.T)
    return out


def dequantize_mxfp8(codes, sf):
    """BF16 = RNE_bf16(E4M3(code) * 2^(sf-127)) [Miles-zh, "高精度反向和去量化反向": the dequantized
    backward consumes a BF16 reconstruction of the exact low-precision forward operands].
    codes [R, C] uint8, sf [R, C/32] uint8 -> bf16 bits [R, C]. The product is exact in float64.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    R, C = codes.shape
    v = e4m3_decode(codes).reshape(R, C // MXFP8_BLOCK, MXFP8_BLOCK)
    e = np.asarray(sf, dtype=np.int64) - 127
    return f64_to_bf16_bits_rne(np.ldexp(v, e[:, :, None]).reshape(R, C))


# ----------------------------------------------------------------------------------------------
# NVFP4
# ----------------------------------------------------------------------------------------------

def nvfp4_token_scale(amax):
    """Coarse FP32 scale for a scope whose max magnitude is ``amax``: RNE_fp32(amax / 2688).

    [Miles-zh, "为什么需要 Blackwell 原生方案？": the coarse FP32 scale maps a tensor or a token into
    NVFP4's representable range; "逐 Token 激活值缩放": one FP32 scale per token, computed online.]
    Reading (the pages give no formula): the scale is a decode multiplier chosen so that amax maps
    onto the largest product of an E2M1 value and an E4M3 block scale, 6 * 448 = 2688. It is the
    correctly rounded fp32 quotient (subnormals kept). See the module docstring for exactness.
    """
    a = np.asarray(amax, dtype=np.float64)
    return (a / NVFP4_RANGE).astype(np.float32)


def pack_e2m1(codes):
    """Pack E2M1 codes [R, C] into bytes [R, C/2]: element 2j -> low nibble, 2j+1 -> high nibble
    (reading; the pages do not fix the nibble order)."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)


def unpack_e2m1(packed):
    p = np.asarray(packed, dtype=np.uint8)
    R, H = p.shape
    out = np.empty((R, 2 * H), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def nvfp4_quantize_rows(x, s):
    """Quantize rows of real matrix x [R, C] in 1x16 blocks, given each row's coarse scale s [R].

    Per block [Miles-zh, "为什么需要 Blackwell 原生方案？" (NVFP4: 16 E2M1 values share an E4M3 block
    scale, rounded to the nearest representable value); NVFP4-ru, second paragraph (block of 16,
    E4M3 block scale, extra FP32 level)]; values use round-to-nearest-even with saturation (method
    statement):
      sf   = E4M3_RNE_satfinite(amax_block / (6 * s))      (s == 0 -> sf = 0)
      code = E2M1_RNE_satfinite(x / (E4M3(sf) * s))        (E4M3(sf) == 0 -> signed zero)
    Returns (packed codes uint8 [R, C/2], sf uint8 [R, C/16]).
    """
    x = np.asarray(x, dtype=np.float64)
    R, C = x.shape
    if C % NVFP4_BLOCK:
        raise ValueError("row length must be a multiple of 16")
    s64 = np.asarray(s, dtype=np.float32).astype(np.float64).reshape(R, 1, 1)
    blocks = x.reshape(R, C // NVFP4_BLOCK, NVFP4_BLOCK)
    amax_b = np.abs(blocks).max(axis=2, keepdims=True) if C else np.zeros((R, 0, 1))
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s64 > 0, amax_b / (6.0 * s64), 0.0)
    sf = round_to_e4m3(q)                                   # non-negative: codes 0x00..0x7E
    d = e4m3_decode(sf) * s64                               # exact: 4 x 24 significant bits
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(d > 0, blocks / np.where(d > 0, d, 1.0), blocks * 0.0)  # 0*x keeps x's sign
    codes = round_to_e2m1(y).reshape(R, C)
    return pack_e2m1(codes), sf.reshape(R, C // NVFP4_BLOCK)


def nvfp4_quantize_per_token(x_bits):
    """Per-token NVFP4 of a bf16 matrix X [T, K]: one FP32 scale per row (token).

    [Miles-zh, "逐 Token 激活值缩放": per-tensor scaling makes a token's representation depend on
    the batch, so the recipe computes one FP32 activation scale per token online, and the same
    call that emits packed FP4 activations and E4M3 block scales also returns the per-token FP32
    scales; Miles-fr, "Un quantificateur partagé est le véritable mécanisme", same.]
    Returns (packed [T, K/2] uint8, sf [T, K/16] uint8, s_tok [T] float32).
    """
    x = _finite_bf16(x_bits)
    T, K = x.shape
    amax = np.abs(x).max(axis=1) if K else np.zeros(T)
    s_tok = nvfp4_token_scale(amax)
    q, sf = nvfp4_quantize_rows(x, s_tok)
    return q, sf, s_tok


def nvfp4_quantize_weights(w_bits):
    """NVFP4 expert weights W [E, K, N] (bf16, Y = X W): one FP32 scale per expert matrix, 1x16
    blocks along K, stored K-major as [E, N, K/2] / [E, N, K/16].

    [Miles-zh, "逐 Token 激活值缩放": SwiGLU gate and up projections are fused into one GEMM, so
    both must share one FP32 scale, which the NVFP4 export enforces by quantizing the gate/up pair
    together; "方案 1" / Miles-fr: microscaling blocks follow the GEMM reduction dimension (K);
    Miles-zh, "移除额外的 BF16 权重副本": the recipe's weight layout is 1-D 1x16.] Reading: the
    coarse-scale scope is the whole [K, N] expert matrix (gate and up concatenated along N), so
    the gate/up pair shares it by construction.
    Returns (packed [E, N, K/2], sf [E, N, K/16], s_w [E] float32).
    """
    w = _finite_bf16(w_bits)
    E, K, N = w.shape
    amax = np.abs(w).reshape(E, -1).max(axis=1) if K * N else np.zeros(E)
    s_w = nvfp4_token_scale(amax)
    wt = np.ascontiguousarray(w.transpose(0, 2, 1)).reshape(E * N, K)
    q, sf = nvfp4_quantize_rows(wt, np.repeat(s_w, N))
    return q.reshape(E, N, K // 2), sf.reshape(E, N, K // NVFP4_BLOCK), s_w


def dequantize_nvfp4(packed, sf, s):
    """BF16 = RNE_bf16(E2M1(code) * E4M3(sf) * s) for packed rows [R, C/2], sf [R, C/16] and a
    coarse scale per row s [R] [Miles-zh, "高精度反向和去量化反向"]. The triple product has at most
    2 + 4 + 24 significant bits, so it is exact in float64 and rounded once to bf16.
    """
    codes = unpack_e2m1(packed)
    R, C = codes.shape
    v = e2m1_decode(codes).reshape(R, C // NVFP4_BLOCK, NVFP4_BLOCK)
    sc = e4m3_decode(sf)[:, :, None] * np.asarray(s, dtype=np.float32).astype(np.float64).reshape(R, 1, 1)
    return f64_to_bf16_bits_rne((v * sc).reshape(R, C))
