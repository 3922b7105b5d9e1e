"""SwiGLU of a gate||up activation pair, as the bf16 input of the down projection.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages' MoE experts are SwiGLU layers whose gate and up projections run as one fused GEMM
[Miles-zh, "逐 Token 激活值缩放": gate and up are fused into one GEMM and share one FP32 scale;
Miles-fr, same paragraph], and the per-token FP32 scaling belongs inside the quantization kernel
rather than a separate op [Miles-zh, "结果" (the training-side gap comes from an unfused scaling
op); "逐 Token 激活值缩放" (one call emits FP4 values, E4M3 block scales and per-token scales)].
The pages do not spell out the activation's arithmetic. Reading taken: SwiGLU(g, u) = silu(g) * u
with silu(g) = g / (1 + exp(-g)) (Shazeer, "GLU Variants Improve Transformer", 2020), gate = the
first half of the fused GEMM's output columns and up = the second half, computed in float32 and
rounded once to bf16 -- the value an unfused path would store as the down projection's input.

Because the result is rounded to bf16 and then quantized, the float32 steps must be identical on
both sides of a bit-exact comparison, and a library exp cannot be reproduced here. The steps are
float32 operations with one rounding each (no fused multiply-add), on an exp of our own:

  x = -g, clamped to [-87, 300]. Below -87, exp(x) < 2^-125 and d = 1 + exp(x) is exactly 1 in
      float32 either way; above 300 the result rounds to a signed zero either way (|g u| < 2^256
      and exp(300) > 2^432, so |h| < 2^-176), so the clamp never changes a result;
  n = nearest integer to x * log2(e), by adding and subtracting 1.5 * 2^23 (ties to even);
  r = (x - n * ln2_hi) - n * ln2_lo  (Cody and Waite's two-constant reduction, W. J. Cody and
      W. Waite, "Software Manual for the Elementary Functions", 1980; ln2_hi = 0x3F317200 has 16
      trailing zero bits and |n| <= 433, so n * ln2_hi is exact);
  p = 1 + r + r^2/2! + ... + r^6/6!  (Taylor polynomial, Horner order; |r| <= ln2/2 keeps the
      truncation below 1.2e-7 relative);
  exp(x) ~ p * 2^n, kept as the pair (p, n).

The exponent range of exp(-g), d and s is unbounded: float32 significands, one rounding each, no
overflow or underflow in these intermediates. Only the final product is rounded to the float32
format itself (gradual underflow), then to bf16. Concretely:

  x <= 87 (2^n is a normal float32): e = p * 2^n, d = 1 + e, s = g / d (IEEE division),
      h32 = s * u -- plain IEEE float32 steps; none of e, d, s leaves the normal range or is
      rounded as a subnormal (for subnormal g, s = g / 2 exactly).
  x > 87 (exp(-g) > 2^125): d = p * 2^n exactly (1 lies far below half an ulp of it), so
      s = RN(g / p) * 2^-n. It is formed as q = RN((g * 2^-16) / p) (the power-of-two factor keeps
      the quotient finite for any bf16 g and changes no rounding), and h32 = RN_f32(q * u *
      2^(16 - n)), one rounding of an exact product (in float64: a 24-bit by 8-bit product times a
      power of two). On the overlap both forms give the same h32.

Then h = RN_bf16(h32).

A plain float32 evaluation would instead overflow exp(-g) to +inf for g < -88.72 and return a
signed zero there, which departs from silu(g) * u when |u| is large (g = -90, u = 1e30 gives
-7.4e-8, not -0); this reading keeps the definition for every finite input whose result is finite.

Pinning: ``tests/test_oracle_swiglu.py`` checks (p, n) against math.exp within 4 float32 ulp on a
dense grid over [-87, 300] (measured worst case below 3), the SwiGLU against float64 silu(g) * u
within one bf16 rounding plus the float32 error for every bf16 gate in [-bf16 max, 100] with large
and small |u|, and the closed-form special cases (g = 0, large positive and negative g).
"""

import numpy as np

F = np.float32
_L2E = F(1.4426950408889634)          # log2(e)
_LN2_HI = F(0.693145751953125)        # 0x3F317200
_LN2_LO = F(0.6931471805599453 - 0.693145751953125)
_MAGIC = F(12582912.0)                # 1.5 * 2^23
_C = [F(1.0 / 720.0), F(1.0 / 120.0), F(1.0 / 24.0), F(1.0 / 6.0), F(0.5), F(1.0), F(1.0)]
X_MIN, X_MAX = F(-87.0), F(300.0)
X_NORMAL = F(87.0)                    # x <= 87: 2^n (n <= 126) is a normal float32
G_SHIFT = 16                          # g * 2^-16 in the quotient of the x > 87 form


def exp_parts(x):
    """(p, n) with exp(x) ~ p * 2^n for float32 x clamped to [X_MIN, X_MAX]: p float32 (in about
    [0.7, 1.42]), n int64. The steps of the module docstring."""
    x = np.asarray(x, dtype=F)
    with np.errstate(over="ignore", under="ignore"):
        x = np.minimum(np.maximum(x, X_MIN), X_MAX)
        t = (x * _L2E).astype(F)
        n = ((t + _MAGIC).astype(F) - _MAGIC).astype(F)
        r = ((x - (n * _LN2_HI).astype(F)).astype(F) - (n * _LN2_LO).astype(F)).astype(F)
        p = _C[0]
        for c in _C[1:]:
            p = ((p * r).astype(F) + c).astype(F)
    return np.asarray(p, dtype=F), np.asarray(n, dtype=np.float64).astype(np.int64)


def exp_f32(x):
    """exp(x) as a float32 for x <= 87, where p * 2^n is a normal float32 (x < -87 gives exp(-87))."""
    x = np.asarray(x, dtype=F)
    if np.any(x > X_NORMAL):
        raise ValueError("exp_f32 covers x <= 87; use exp_parts above")
    p, n = exp_parts(x)
    two_n = ((n + 127).astype(np.uint32) << 23).view(F)
    with np.errstate(over="ignore", under="ignore"):
        return (p * two_n).astype(F)


def swiglu_f32(g, u):
    """float32 h32 of the module docstring from float32 g and u (same shape)."""
    g = np.asarray(g, dtype=F)
    u = np.asarray(u, dtype=F)
    x = (-g).astype(F)
    p, n = exp_parts(x)
    big = x > X_NORMAL
    with np.errstate(over="ignore", under="ignore", invalid="ignore", divide="ignore"):
        # x <= 87: IEEE float32 steps
        n_small = np.where(big, 0, n)
        two_n = ((n_small + 127).astype(np.uint32) << 23).view(F)
        e = (p * two_n).astype(F)
        d = (F(1.0) + e).astype(F)
        s = (g / d).astype(F)
        h_small = (s * u).astype(F)
        # x > 87: d = p 2^n exactly; one rounding of q u 2^(16 - n) to float32
        q = ((g * F(2.0 ** -G_SHIFT)).astype(F) / p).astype(F)
        h64 = q.astype(np.float64) * u.astype(np.float64) * np.ldexp(1.0, (G_SHIFT - n).astype(np.int32))
        h_big = h64.astype(F)
    return np.where(big, h_big, h_small).astype(F)


def swiglu_bf16_bits(gate_bits, up_bits):
    """bf16 bits of RN_bf16(silu(g) * u), elementwise, from bf16 bits of g and u (same shape)."""
    g = (np.asarray(gate_bits, dtype=np.uint16).astype(np.uint32) << 16).view(F)
    u = (np.asarray(up_bits, dtype=np.uint16).astype(np.uint32) << 16).view(F)
    h32 = swiglu_f32(g, u)
    from .formats import f64_to_bf16_bits_rne
    return f64_to_bf16_bits_rne(h32.astype(np.float64))


def swiglu_rows(gate_up_bits):
    """SwiGLU of a fused gate||up activation [R, 2I] (bf16 bits): gate = columns [0, I), up =
    columns [I, 2I). Returns bf16 bits [R, I]."""
    a = np.asarray(gate_up_bits, dtype=np.uint16)
    if a.ndim != 2 or a.shape[1] % 2:
        raise ValueError("expected [R, 2I]")
    I = a.shape[1] // 2
    return swiglu_bf16_bits(a[:, :I], a[:, I:])
