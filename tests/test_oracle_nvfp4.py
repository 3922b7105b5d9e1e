"""Pins for the oracle's per-token NVFP4 quantizer (no GPU): the hand-worked token, the block-amax
invariant of the NVFP4 pretraining summary, and per-token invariance under batch changes."""
import numpy as np
import torch

import oracle
from tests._golden import bf16_exact_bits, hexbytes, load


def _bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_hand_worked_token():
    g = load("nvfp4_token.json")
    row = np.concatenate([bf16_exact_bits(b) for b in g["row_values"]]).reshape(1, -1)
    q, sf, s = oracle.nvfp4_quantize_per_token(row)
    assert s[0] == np.float32(g["s_tok"])
    assert np.array_equal(sf[0], hexbytes(g["sf"]))
    assert np.array_equal(q[0], np.concatenate([hexbytes(p) for p in g["packed"]]))


def test_block_amax_encodes_as_six_when_scale_is_normal():
    # NVFP4-ru: at least 6.25% of each block (its amax, 1 of 16) is represented near FP8 precision:
    # with an E4M3-normal block scale the amax element maps onto E2M1's largest value.
    rng = np.random.default_rng(7)
    x = rng.standard_normal((256, 512)) * np.exp(rng.uniform(-8, 8, (256, 1))) * \
        np.exp(rng.uniform(-4, 0, (256, 32)).repeat(16, axis=1))
    bits = _bits(x)
    q, sf, s = oracle.nvfp4_quantize_per_token(bits)
    codes = oracle.unpack_e2m1(q).reshape(256, 32, 16)
    xb = np.abs(oracle.bf16_bits_to_f64(bits)).reshape(256, 32, 16)
    arg = xb.argmax(axis=2)
    amax_code = np.take_along_axis(codes, arg[:, :, None], axis=2)[:, :, 0] & 7
    normal = (sf >= 0x08) & (sf <= 0x7E)
    assert normal.sum() > 1000
    assert np.all(amax_code[normal] == 7)


def test_token_amax_block_gets_top_scale():
    # s = RN(amax/2688) => the block holding the token amax gets sf = 448 (0x7E) when s is normal.
    rng = np.random.default_rng(8)
    x = rng.standard_normal((512, 256)) * np.exp(rng.uniform(-30, 30, (512, 1)))
    bits = _bits(x)
    q, sf, s = oracle.nvfp4_quantize_per_token(bits)
    xb = np.abs(oracle.bf16_bits_to_f64(bits))
    blk = xb.argmax(axis=1) // 16
    assert np.all(sf[np.arange(512), blk] == 0x7E)


def test_per_token_invariance_under_batch_changes():
    # Miles-zh "逐 Token 激活值缩放": a token's quantized bits must not depend on the rest of the batch.
    rng = np.random.default_rng(9)
    x = _bits(rng.standard_normal((64, 256)) * np.exp(rng.uniform(-5, 5, (64, 1))))
    q, sf, s = oracle.nvfp4_quantize_per_token(x)
    perm = rng.permutation(64)
    q2, sf2, s2 = oracle.nvfp4_quantize_per_token(x[perm])
    assert np.array_equal(q2, q[perm]) and np.array_equal(sf2, sf[perm]) and np.array_equal(s2, s[perm])
    other = _bits(rng.standard_normal((64, 256)) * 1e4)
    mixed = np.concatenate([x[:10], other[:30]])
    q3, sf3, s3 = oracle.nvfp4_quantize_per_token(mixed)
    assert np.array_equal(q3[:10], q[:10]) and np.array_equal(sf3[:10], sf[:10])
    assert np.array_equal(s3[:10], s[:10])
    q4, sf4, s4 = oracle.nvfp4_quantize_per_token(x[5:6])
    assert np.array_equal(q4[0], q[5]) and np.array_equal(sf4[0], sf[5]) and s4[0] == s[5]


def test_zero_and_max_rows():
    z = np.zeros((2, 32), dtype=np.uint16)
    z[1, 3] = 0x8000                               # -0
    q, sf, s = oracle.nvfp4_quantize_per_token(z)
    assert np.all(s == 0) and not sf.any()
    codes = oracle.unpack_e2m1(q)
    assert codes[1, 3] == 8 and (np.delete(codes.reshape(-1), 32 + 3) == 0).all()
    m = np.full((1, 32), 0x7F7F, dtype=np.uint16)
    q, sf, s = oracle.nvfp4_quantize_per_token(m)
    assert np.all(sf == 0x7E) and np.all(oracle.unpack_e2m1(q) == 7)


def test_weight_scope_is_whole_expert_matrix():
    # Miles-zh: gate and up share one FP32 scale because they feed one fused GEMM.
    rng = np.random.default_rng(10)
    w = rng.standard_normal((3, 64, 48)) * 0.02
    w[1, :, :24] *= 50                                   # gate half of expert 1 much larger
    bits = _bits(w)
    q, sf, s_w = oracle.nvfp4_quantize_weights(bits)
    xb = np.abs(oracle.bf16_bits_to_f64(bits))
    for e in range(3):
        assert s_w[e] == np.float32(xb[e].max() / 2688.0)
        # the scope's rows are the N columns of W[e], quantized along K with the shared scale
        qe, sfe = oracle.nvfp4_quantize_rows(oracle.bf16_bits_to_f64(bits[e]).T, np.full(48, s_w[e]))
        assert np.array_equal(q[e], qe) and np.array_equal(sf[e], sfe)
    # quantizing gate and up separately would give different scales (and bytes) for expert 1
    _, _, s_gate = oracle.nvfp4_quantize_weights(np.ascontiguousarray(bits[1:2, :, :24]))
    _, _, s_up = oracle.nvfp4_quantize_weights(np.ascontiguousarray(bits[1:2, :, 24:]))
    assert s_gate[0] == s_w[1] and s_up[0] != s_w[1]
