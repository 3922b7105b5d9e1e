"""Every NVFP4 coarse scale through the GPU quantizers, against the oracle byte for byte.

[Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本", section "比特精确量化器合约":
the quantizer must match its reference byte for byte on random, boundary, zero and max inputs.]
The quantizers decide each rounding with a per-scope table (the coarse scale s = RN(amax / 2688)
of a token row or of an expert matrix) and take one of three encode paths per scope. Here one scope
is made for every positive finite bf16 amax (32639 of them), and its other elements sit on, and one
bf16 ulp either side of, the E2M1 decision thresholds m * E4M3(sf) * s of their blocks, with block
maxima spread over 16 binades, so that every scope's table build, its product-path check and the
encoding of each block meet values at their decision boundaries.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


@pytest.fixture(scope="module")
def nvq():
    import nvfp4_quantization_block_gb300 as m
    return m


def _scope_rows(length, seed, frac_step):
    """bf16 bits [32639, length]: row r's amax is the r-th positive finite bf16 value; block b's max
    is that amax times 2^(-b * frac_step) (bf16-rounded); the other 15 elements of each block are
    the bf16 values at and next to the block's E2M1 thresholds (never above its max), signs random,
    positions rotated per row."""
    amax_bits = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)
    R, nb = len(amax_bits), length // 16
    A = oracle.bf16_bits_to_f64(amax_bits)
    s = oracle.nvfp4_token_scale(A).astype(np.float64)
    frac = 2.0 ** (-frac_step * np.arange(nb))
    a_bits = oracle.f64_to_bf16_bits_rne(A[:, None] * frac[None, :])
    a_bits[:, 0] = amax_bits
    a = oracle.bf16_bits_to_f64(a_bits)                                   # block maxima [R, nb]
    with np.errstate(divide="ignore", invalid="ignore"):
        sf = oracle.round_to_e4m3(np.where(s[:, None] > 0, a / (6.0 * s[:, None]), 0.0))
    v = oracle.e4m3_decode(sf)
    t = MIDPOINTS[None, None, :] * v[:, :, None] * s[:, None, None]         # thresholds [R, nb, 7]
    tb = oracle.f64_to_bf16_bits_rne(t).astype(np.int32)
    cand = np.concatenate([tb - 1, tb, tb + 1], axis=2).clip(0, 0x7F7F)    # [R, nb, 21]
    cv = np.minimum(oracle.bf16_bits_to_f64(cand.astype(np.uint16)), a[:, :, None])
    cbits = oracle.f64_to_bf16_bits_rne(cv)
    rng = np.random.default_rng(seed)
    k = (np.arange(15)[None, None, :] + np.arange(R)[:, None, None] + np.arange(nb)[None, :, None]) % 21
    others = np.take_along_axis(cbits, k, axis=2)                          # [R, nb, 15]
    others = others | (rng.integers(0, 2, others.shape).astype(np.uint16) << 15)
    blocks = np.concatenate([a_bits[:, :, None], others], axis=2)         # [R, nb, 16]
    rot = (np.arange(R)[:, None, None] + np.arange(16)[None, None, :]) % 16
    blocks = np.take_along_axis(blocks, np.broadcast_to(rot, blocks.shape), axis=2)
    return blocks.reshape(R, nb * 16)


@pytest.mark.parametrize("length,layout", [(256, "mma"), (1056, "canonical")])
def test_per_token_every_coarse_scale(nvq, length, layout):
    # 256: two rows per warp (boundary comparisons); 1056: one row per warp, product-path check
    bits = _scope_rows(length, seed=length, frac_step=1.0 if length == 256 else 0.25)
    q, sf, s = nvq.nvfp4_quantize_per_token(workloads.from_bits(bits, "cuda"), sf_layout=layout)
    torch.cuda.synchronize()
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(bits)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    bad = np.nonzero((q.cpu().numpy() != q_ref).any(axis=1))[0]
    assert len(bad) == 0, f"{len(bad)} rows differ, first amax bits {bad[:8] + 1}"
    got_sf = sf.cpu().numpy()
    want_sf = sf_ref if layout == "canonical" else oracle.sf_to_mma_layout(sf_ref)
    assert np.array_equal(got_sf.reshape(want_sf.shape), want_sf)


def test_weights_every_coarse_scale(nvq):
    # 32639 experts of [K = 16, N = 8]: expert e's amax is the e-th positive bf16 value; each of its
    # eight K-blocks (one per output column) is built as above
    rows = _scope_rows(128, seed=7, frac_step=1.0)                       # [E, 8 blocks of 16]
    E = rows.shape[0]
    w = np.ascontiguousarray(rows.reshape(E, 8, 16).transpose(0, 2, 1))  # [E, K=16, N=8]
    qT, sfT, s_w = nvq.nvfp4_quantize_weights(workloads.from_bits(w, "cuda"), sf_layout="canonical")
    torch.cuda.synchronize()
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_weights(w)
    assert np.array_equal(s_w.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    bad = np.nonzero((qT.cpu().numpy().reshape(E, -1) != q_ref.reshape(E, -1)).any(axis=1))[0]
    assert len(bad) == 0, f"{len(bad)} experts differ, first amax bits {bad[:8] + 1}"
    assert np.array_equal(sfT.cpu().numpy().reshape(sf_ref.shape), sf_ref)
