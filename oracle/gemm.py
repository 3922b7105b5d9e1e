"""Block-scaled grouped GEMM over routed MoE experts, in float64 on dequantized operands.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Definition (method statement; [Miles-zh, "方案 1：端到端 MXFP8 强化学习": rollout, forward, weight-
gradient and data-gradient GEMMs all use MXFP8; "方案 2 / 逐 Token 激活值缩放": NVFP4 MoE expert GEMMs
with per-token activation scales; "结果": the fused per-token NVFP4 GEMM applies the FP32 scaling in
the kernel epilogue]). With deq(q) = element value x block scale (E8M0 power of two for MXFP8, E4M3
for NVFP4, the coarse FP32 scales kept apart):

  mode "m" (forward / data gradient; rows of A grouped by expert, offsets o[0..E]):
      D[i, j] = s_a[i] * s_b[e] * sum_k deq(A)[i, k] * deq(B[e])[j, k]     for o[e] <= i < o[e+1]
  mode "k" (weight gradient; the reduction runs over the expert's rows):
      D[e, i, j] = s_a * s_b * sum_{o[e] <= k < o[e+1]} deq(A)[i, k] * deq(B)[j, k]

Both operands are K-major (the reduction index is the contiguous one), as the blocks must follow the
reduction dimension [Miles-fr, "Un quantificateur partagé est le véritable mécanisme"]. Missing s_a
or s_b mean 1. The tolerance the GPU must meet is |D_gpu - D| <= 2e-3 * sum_k |s_a s_b deq(A) deq(B)|
(method statement); ``bound`` returns that sum. np.matmul is the library primitive; everything else
is written out. Pinned by tests/test_oracle_gemm.py (brute-force loops on tiny shapes, the plain
FP8 special case with unit scales, exact integer products).
"""

import numpy as np

from .formats import e2m1_decode, e4m3_decode
from .quant import MXFP8_BLOCK, NVFP4_BLOCK, unpack_e2m1


def deq_operand(fmt, q, sf):
    """Dequantize a K-major operand to float64 without its coarse FP32 scale.

    fmt "mxfp8": q [R, K] E4M3 codes, sf [R, K/32] E8M0 -> E4M3(q) * 2^(sf-127).
    fmt "nvfp4": q [R, K/2] packed E2M1, sf [R, K/16] E4M3 -> E2M1(q) * E4M3(sf).
    """
    if fmt == "mxfp8":
        v = e4m3_decode(q)
        R, K = v.shape
        e = np.asarray(sf, dtype=np.int64) - 127
        return np.ldexp(v.reshape(R, K // MXFP8_BLOCK, MXFP8_BLOCK), e[:, :, None]).reshape(R, K)
    if fmt == "nvfp4":
        v = e2m1_decode(unpack_e2m1(q))
        R, K = v.shape
        s = e4m3_decode(sf)
        return (v.reshape(R, K // NVFP4_BLOCK, NVFP4_BLOCK) * s[:, :, None]).reshape(R, K)
    raise ValueError(fmt)


def _scales(s, n):
    if s is None:
        return np.ones(n)
    return np.asarray(s, dtype=np.float32).astype(np.float64).reshape(-1)


def grouped_gemm_reference(mode, a, b, offsets, s_a=None, s_b=None):
    """Full float64 grouped GEMM on dequantized operands (see module docstring).

    mode "m": a [M, K], b [E, N, K] (float64, from ``deq_operand``), offsets [E+1];
              returns (D [M, N], bound [M, N]); rows outside every group are NaN.
    mode "k": a [Ma, Ktot], b [Nb, Ktot]; returns (D [E, Ma, Nb], bound [E, Ma, Nb]).
    """
    o = np.asarray(offsets, dtype=np.int64)
    E = len(o) - 1
    if mode == "m":
        M, K = a.shape
        N = b.shape[1]
        sa = _scales(s_a, M)
        sb = _scales(s_b, E)
        D = np.full((M, N), np.nan)
        B = np.full((M, N), np.nan)
        for e in range(E):
            r0, r1 = o[e], o[e + 1]
            if r1 <= r0:
                continue
            scale = sa[r0:r1, None] * sb[e]
            D[r0:r1] = scale * (a[r0:r1] @ b[e].T)
            B[r0:r1] = np.abs(scale) * (np.abs(a[r0:r1]) @ np.abs(b[e]).T)
        return D, B
    if mode == "k":
        Ma = a.shape[0]
        Nb = b.shape[0]
        sa = 1.0 if s_a is None else float(np.float32(s_a))
        sb = 1.0 if s_b is None else float(np.float32(s_b))
        D = np.zeros((E, Ma, Nb))
        B = np.zeros((E, Ma, Nb))
        for e in range(E):
            k0, k1 = o[e], o[e + 1]
            D[e] = sa * sb * (a[:, k0:k1] @ b[:, k0:k1].T)
            B[e] = abs(sa * sb) * (np.abs(a[:, k0:k1]) @ np.abs(b[:, k0:k1]).T)
        return D, B
    raise ValueError(mode)


def grouped_gemm_entries(mode, a_rows, b_rows, k_ranges, scale):
    """Selected output entries, one dot product each (for large shapes).

    a_rows [S, K] and b_rows [S, K] are the dequantized operand rows that meet at each sampled
    output, k_ranges [S, 2] the reduction range of each (the whole K in mode "m", the expert's
    segment in mode "k"), scale [S] the product of the FP32 scales. Returns (D [S], bound [S]).
    """
    S = a_rows.shape[0]
    D = np.empty(S)
    Bd = np.empty(S)
    for t in range(S):
        k0, k1 = int(k_ranges[t, 0]), int(k_ranges[t, 1])
        pa = a_rows[t, k0:k1]
        pb = b_rows[t, k0:k1]
        D[t] = scale[t] * np.dot(pa, pb)
        Bd[t] = abs(scale[t]) * np.dot(np.abs(pa), np.abs(pb))
    return D, Bd
