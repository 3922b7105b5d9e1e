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
both sides of a bit-exact comparison, and a library exp cannot be reproduced here. The exp is
therefore our own, in plain float32 operations with one rounding each (no fused multiply-add):
  x clamped to [-87, 88] (so 2^n below stays a normal float);
  n = nearest integer to x * log2(e), by adding and subtracting 1.5 * 2^23 (ties to even);
  r = (x - n * ln2_hi) - n * ln2_lo  (Cody and Waite's two-constant reduction, W. J. Cody and
      W. Waite, "Software Manual for the Elementary Functions", 1980; ln2_hi = 0x3F317200 has 16
      trailing zero bits, so n * ln2_hi is exact);
  p = 1 + r + r^2/2! + ... + r^6/6!  (Taylor polynomial, Horner order; |r| <= ln2/2 keeps the
      truncation below 1.2e-7 relative);
  exp(x) ~ p * 2^n.
Then d = 1 + e, s = g / d (IEEE division), p = s * u, h = RN_bf16(p).

Pinning: ``tests/test_oracle_swiglu.py`` checks the exp against math.exp within 2 float32 ulp on
a dense grid, the SwiGLU against float64 silu(g) * u within one bf16 rounding plus the float32
error, and the closed-form special cases (g = 0, large positive and negative g).
"""

import numpy as np

F = np.float32
_L2E = F(1.4426950408889634)          # log2(e)
_LN2_HI = F(0.693145751953125)        # 0x3F317200
_LN2_LO = F(0.6931471805599453 - 0.693145751953125)
_MAGIC = F(12582912.0)                # 1.5 * 2^23
_C = [F(1.0 / 720.0), F(1.0 / 120.0), F(1.0 / 24.0), F(1.0 / 6.0), F(0.5), F(1.0), F(1.0)]
X_MIN, X_MAX = F(-87.0), F(88.0)


def exp_f32(x):
    """exp(x) for float32 x by the steps in the module docstring; float32 result."""
    x = np.asarray(x, dtype=F)
    with np.errstate(over="ignore", under="ignore"):
        x = np.minimum(np.maximum(x, X_MIN), X_MAX)
        t = (x * _L2E).astype(F)
        n = ((t + _MAGIC).astype(F) - _MAGIC).astype(F)
        r = ((x - (n * _LN2_HI).astype(F)).astype(F) - (n * _LN2_LO).astype(F)).astype(F)
        p = _C[0]
        for c in _C[1:]:
            p = ((p * r).astype(F) + c).astype(F)
        two_n = ((n.astype(np.int32) + 127).astype(np.uint32) << 23).view(F)
        return (p * two_n).astype(F)


def swiglu_bf16_bits(gate_bits, up_bits):
    """bf16 bits of RN_bf16(silu(g) * u), elementwise, from bf16 bits of g and u (same shape)."""
    g = (np.asarray(gate_bits, dtype=np.uint16).astype(np.uint32) << 16).view(F)
    u = (np.asarray(up_bits, dtype=np.uint16).astype(np.uint32) << 16).view(F)
    with np.errstate(over="ignore", under="ignore"):
        e = exp_f32((-g).astype(F))
        d = (F(1.0) + e).astype(F)
        s = (g / d).astype(F)
        p = (s * u).astype(F)
    from .formats import f64_to_bf16_bits_rne
    return f64_to_bf16_bits_rne(p.astype(np.float64))


def swiglu_rows(gate_up_bits):
    """SwiGLU of a fused gate||up activation [R, 2I] (bf16 bits): gate = columns [0, I), up =
    columns [I, 2I). Returns bf16 bits [R, I]."""
    a = np.asarray(gate_up_bits, dtype=np.uint16)
    if a.ndim != 2 or a.shape[1] % 2:
        raise ValueError("expected [R, 2I]")
    I = a.shape[1] // 2
    return swiglu_bf16_bits(a[:, :I], a[:, I:])
