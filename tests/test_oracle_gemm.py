"""Pins for the oracle's grouped GEMM (no GPU): pure-Python brute force on tiny shapes, the plain
FP8 matmul special case (unit E8M0 scales, decoded by torch), exact integer products, and the
relation of the two modes (weight gradient == per-expert transpose products)."""
import numpy as np
import torch

import oracle


def _bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _brute(a, b, offsets, s_a, s_b):
    M, K = a.shape
    N = b.shape[1]
    D = [[None] * N for _ in range(M)]
    for e in range(len(offsets) - 1):
        for i in range(offsets[e], offsets[e + 1]):
            for j in range(N):
                acc = 0.0
                for k in range(K):
                    acc += float(a[i, k]) * float(b[e, j, k])
                D[i][j] = acc * float(s_a[i]) * float(s_b[e])
    return D


def test_mode_m_matches_brute_force_nvfp4():
    rng = np.random.default_rng(0)
    E, N, K = 3, 5, 32
    offsets = np.array([0, 2, 2, 7])
    x = _bits(rng.standard_normal((7, K)) * np.exp(rng.uniform(-3, 3, (7, 1))))
    qa, sfa, sa = oracle.nvfp4_quantize_per_token(x)
    w = _bits(rng.standard_normal((E, K, N)) * 0.02)
    qb, sfb, sb = oracle.nvfp4_quantize_weights(w)
    a = oracle.deq_operand("nvfp4", qa, sfa)
    b = np.stack([oracle.deq_operand("nvfp4", qb[e], sfb[e]) for e in range(E)])
    D, bound = oracle.grouped_gemm_reference("m", a, b, offsets, sa, sb)
    ref = _brute(a, b, offsets, sa.astype(np.float64), sb.astype(np.float64))
    for i in range(7):
        for j in range(N):
            assert abs(D[i, j] - ref[i][j]) <= 1e-12 * bound[i, j] + 1e-300
    assert np.all(bound >= np.abs(D) * (1 - 1e-12))


def test_unit_scales_reduce_to_plain_fp8_matmul():
    # E8M0 byte 127 = 2^0: the block-scaled GEMM is an ordinary FP8 x FP8 matmul. Codes decoded by
    # torch's float8_e4m3fn; integer-valued products make the float64 result exact.
    rng = np.random.default_rng(1)
    codes_a = rng.choice(np.arange(0x38, 0x58), (16, 64)).astype(np.uint8)   # 1 .. 15 range
    codes_b = rng.choice(np.arange(0x38, 0x58), (2, 8, 64)).astype(np.uint8)
    codes_a |= (rng.random((16, 64)) < 0.5).astype(np.uint8) << 7
    sfa = np.full((16, 2), 127, np.uint8)
    sfb = np.full((2, 8, 2), 127, np.uint8)
    a = oracle.deq_operand("mxfp8", codes_a, sfa)
    b = np.stack([oracle.deq_operand("mxfp8", codes_b[e], sfb[e]) for e in range(2)])
    D, _ = oracle.grouped_gemm_reference("m", a, b, [0, 5, 16])
    ta = torch.from_numpy(codes_a).view(torch.float8_e4m3fn).double()
    tb = torch.from_numpy(codes_b).view(torch.float8_e4m3fn).double()
    ref = torch.cat([ta[:5] @ tb[0].T, ta[5:] @ tb[1].T]).numpy()
    assert np.array_equal(D, ref)


def test_mode_k_is_per_segment_product():
    rng = np.random.default_rng(2)
    xa = _bits(rng.standard_normal((96, 64)))       # [rows, features]
    dy = _bits(rng.standard_normal((96, 32)) * 1e-3)
    qa = oracle.mxfp8_quantize(xa)
    qd = oracle.mxfp8_quantize(dy)
    A = oracle.deq_operand("mxfp8", qa["q_colT"], qa["sf_colT"])   # [64, 96]
    B = oracle.deq_operand("mxfp8", qd["q_colT"], qd["sf_colT"])   # [32, 96]
    offs = [0, 32, 32, 96]
    D, bound = oracle.grouped_gemm_reference("k", A, B, offs)
    assert np.all(D[1] == 0)
    for e in (0, 2):
        ref = A[:, offs[e]:offs[e + 1]] @ B[:, offs[e]:offs[e + 1]].T
        assert np.allclose(D[e], ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    # one entry by hand
    k0, k1 = offs[2], offs[3]
    assert abs(D[2, 3, 5] - sum(A[3, k] * B[5, k] for k in range(k0, k1))) <= 1e-12 * bound[2, 3, 5]


def test_entries_match_full():
    rng = np.random.default_rng(3)
    a = rng.standard_normal((20, 48))
    b = rng.standard_normal((2, 6, 48))
    D, bound = oracle.grouped_gemm_reference("m", a, b, [0, 11, 20], np.ones(20), np.ones(2))
    ii = np.array([0, 10, 11, 19])
    jj = np.array([5, 0, 3, 2])
    ee = np.array([0, 0, 1, 1])
    d, bd = oracle.grouped_gemm_entries("m", a[ii], b[ee, jj], np.tile([0, 48], (4, 1)), np.ones(4))
    assert np.allclose(d, D[ii, jj], rtol=1e-13) and np.allclose(bd, bound[ii, jj], rtol=1e-13)
