"""GPU parity: the sm_103a quantizers and dequantizer against the CPU oracle, byte for byte.

Input families follow the upstream contract tests described on the pages ("random", "boundary",
"zeros", "maxes" [Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本", section
"比特精确量化器合约"]), at sizes spanning several tiles with ragged tails, in both scale layouts.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvq():
    import nvfp4_quantization_block_gb300 as m
    return m


def _seed(*parts):
    return zlib.crc32(repr(parts).encode()) % 10007


def _np(t):
    return t.detach().cpu().numpy()


def _bits_of(x_f64):
    """Host bf16 bits of float64 values (exactly representable ones stay exact)."""
    return oracle.f64_to_bf16_bits_rne(np.asarray(x_f64, dtype=np.float64))


def _dev(bits):
    return workloads.from_bits(bits, "cuda")


# ------------------------------------------------------------------------------------------------
# input families
# ------------------------------------------------------------------------------------------------
def family(name, shape, seed=0):
    rng = np.random.default_rng(seed)
    R, C = shape
    if name == "random":
        x = rng.standard_normal(shape) * np.exp(rng.uniform(-12, 12, (R, 1)))
        x *= np.where(rng.random(shape) < 0.01, 100.0, 1.0)
        return _bits_of(x)
    if name == "zeros":
        b = np.zeros(shape, dtype=np.uint16)
        b[rng.random(shape) < 0.3] = 0x8000          # negative zeros keep their sign
        return b
    if name == "maxes":
        b = np.full(shape, 0x7F7F, dtype=np.uint16)
        b[rng.random(shape) < 0.5] |= 0x8000
        return b
    if name == "boundary":
        # values on E4M3 / E2M1 rounding midpoints and their bf16 neighbours, scaled by powers of
        # two and by the "nice" NVFP4 token scale 2^k (token amax 42*2^(k+6)), plus subnormals
        mids4 = (oracle.E4M3_VALUES[:-1] + oracle.E4M3_VALUES[1:]) / 2
        mids2 = (oracle.E2M1_VALUES[:-1] + oracle.E2M1_VALUES[1:]) / 2
        base = np.concatenate([mids4, oracle.E4M3_VALUES, mids2 * 8, mids2 * 11, mids2 * 448, [448, 450, 449.5]])
        v = rng.choice(base, shape) * np.ldexp(1.0, rng.integers(-20, 20, (R, 1)))
        v = oracle.bf16_bits_to_f64(_bits_of(v))
        ulp = np.ldexp(1.0, np.frexp(v)[1] - 8)
        v = v + rng.choice([-1, 0, 0, 0, 1], shape) * ulp
        v *= rng.choice([-1, 1], shape)
        tiny = rng.random(shape) < 0.03
        v[tiny] = rng.integers(1, 200, tiny.sum()) * 2.0 ** -133
        b = _bits_of(v)
        # rows whose amax gives an exact power-of-two token scale
        nice = rng.random(R) < 0.5
        col = rng.integers(0, C, R)
        b[nice, col[nice]] = _bits_of(42.0 * np.ldexp(1.0, rng.integers(-10, 10, nice.sum())))
        return b
    raise ValueError(name)


FAMILIES = ["random", "boundary", "zeros", "maxes"]


# ------------------------------------------------------------------------------------------------
# MXFP8
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("fam", FAMILIES)
@pytest.mark.parametrize("shape", [(256, 512), (320, 416), (96, 64), (32, 32), (416, 1056)])
@pytest.mark.parametrize("layout", ["canonical", "mma"])
def test_mxfp8_row_col_bit_exact(nvq, fam, shape, layout):
    bits = family(fam, shape, seed=_seed(fam, shape))
    ref = oracle.mxfp8_quantize(bits)
    out = nvq.mxfp8_quantize(_dev(bits), sf_layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(_np(out["q_row"]), ref["q_row"])
    assert np.array_equal(_np(out["q_colT"]), ref["q_colT"])
    if layout == "canonical":
        assert np.array_equal(_np(out["sf_row"]).reshape(ref["sf_row"].shape), ref["sf_row"])
        assert np.array_equal(_np(out["sf_colT"]).reshape(ref["sf_colT"].shape), ref["sf_colT"])
    else:
        assert np.array_equal(_np(out["sf_row"]), oracle.sf_to_mma_layout(ref["sf_row"]))
        assert np.array_equal(_np(out["sf_colT"]), oracle.sf_to_mma_layout(ref["sf_colT"]))


@pytest.mark.parametrize("rowwise", [True, False])
def test_mxfp8_deep_grid_staged_path(nvq, rowwise):
    """A grid deeper than two waves (33 x 41 tiles of 128 x 128, ragged in both directions) takes
    the shared-memory staged variant of the kernel; bit-exact against the oracle, both copies."""
    shape = (4128, 5152)
    bits = family("random", shape, seed=17)
    ref = oracle.mxfp8_quantize(bits, rowwise=rowwise)
    o = nvq.mxfp8_quantize(_dev(bits), rowwise=rowwise, sf_layout="mma")
    torch.cuda.synchronize()
    assert np.array_equal(_np(o["q_colT"]), ref["q_colT"])
    assert np.array_equal(_np(o["sf_colT"]), oracle.sf_to_mma_layout(ref["sf_colT"]))
    if rowwise:
        assert np.array_equal(_np(o["q_row"]), ref["q_row"])
        assert np.array_equal(_np(o["sf_row"]), oracle.sf_to_mma_layout(ref["sf_row"]))


@pytest.mark.parametrize("shape,rowwise", [((2048, 5120), False), ((2048, 5632), True)])
def test_mxfp8_one_wave_staged_path(nvq, shape, rowwise):
    """Grids just past one wave of the register variant that fit one wave of the staged variant
    (640 column-only tiles: the dense W_qkv's columnwise copy; 704 row+col tiles) take the staged
    variant on a 152-SM GPU; bit-exact against the oracle either way."""
    bits = family("random", shape, seed=23)
    ref = oracle.mxfp8_quantize(bits, rowwise=rowwise)
    o = nvq.mxfp8_quantize(_dev(bits), rowwise=rowwise, sf_layout="mma")
    torch.cuda.synchronize()
    assert np.array_equal(_np(o["q_colT"]), ref["q_colT"])
    assert np.array_equal(_np(o["sf_colT"]), oracle.sf_to_mma_layout(ref["sf_colT"]))
    if rowwise:
        assert np.array_equal(_np(o["q_row"]), ref["q_row"])
        assert np.array_equal(_np(o["sf_row"]), oracle.sf_to_mma_layout(ref["sf_row"]))


@pytest.mark.parametrize("shape", [(33, 64), (1, 32), (7, 96)])
def test_mxfp8_rowwise_only_ragged_rows(nvq, shape):
    bits = family("random", shape, seed=3)
    ref = oracle.mxfp8_quantize(bits, colwise=False)
    for layout in ("canonical", "mma"):
        out = nvq.mxfp8_quantize(_dev(bits), colwise=False, sf_layout=layout)
        assert np.array_equal(_np(out["q_row"]), ref["q_row"])
        want = ref["sf_row"] if layout == "canonical" else oracle.sf_to_mma_layout(ref["sf_row"])
        assert np.array_equal(_np(out["sf_row"]).reshape(want.shape), want)


def test_mxfp8_columnwise_output_off_the_32_byte_grid(nvq):
    # q_colT 16 bytes past a 32-byte boundary: the columnwise codes take 16-byte stores instead of
    # one 256-bit store per column and block; the bytes are the same
    R, C = 96, 160
    bits = family("random", (R, C), seed=8)
    ref = oracle.mxfp8_quantize(bits)
    buf = torch.empty(C * R + 32, dtype=torch.uint8, device="cuda")
    qT = buf[16:16 + C * R].view(C, R)
    out = nvq.mxfp8_quantize(_dev(bits), sf_layout="canonical", out={"q_colT": qT})
    torch.cuda.synchronize()
    assert np.array_equal(_np(out["q_colT"]), ref["q_colT"])
    assert np.array_equal(_np(out["sf_colT"]).reshape(ref["sf_colT"].shape), ref["sf_colT"])
    assert np.array_equal(_np(out["q_row"]), ref["q_row"])


def test_mxfp8_strided_input(nvq):
    bits = family("random", (128, 256), seed=4)
    big = torch.zeros((128, 320), dtype=torch.bfloat16, device="cuda")
    big[:, :256] = _dev(bits)
    ref = oracle.mxfp8_quantize(bits)
    out = nvq.mxfp8_quantize(big[:, :256], sf_layout="canonical")
    assert np.array_equal(_np(out["q_row"]), ref["q_row"])
    assert np.array_equal(_np(out["q_colT"]), ref["q_colT"])


# ------------------------------------------------------------------------------------------------
# NVFP4 per token
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("fam", FAMILIES)
@pytest.mark.parametrize("shape", [(300, 768), (257, 2048), (64, 4096), (5, 48), (130, 272)])
@pytest.mark.parametrize("layout", ["canonical", "mma"])
def test_nvfp4_per_token_bit_exact(nvq, fam, shape, layout):
    bits = family(fam, shape, seed=_seed(fam, shape, 1))
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(bits)
    q, sf, s = nvq.nvfp4_quantize_per_token(_dev(bits), sf_layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(_np(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(_np(q), q_ref)
    want = sf_ref if layout == "canonical" else oracle.sf_to_mma_layout(sf_ref)
    assert np.array_equal(_np(sf).reshape(want.shape), want)


@pytest.mark.parametrize("shape", [(16001, 256), (7500, 1040)])
def test_nvfp4_per_token_many_row_groups_per_warp(nvq, shape):
    """More row groups than a 152-SM GPU holds resident warps, so each warp takes two or three in
    turn and the last turn is ragged (two rows per warp at 256 columns, one at 1040): every byte
    equals the oracle's in both scale layouts."""
    bits = family("random", shape, seed=_seed("random", shape, 7))
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(bits)
    for layout in ("canonical", "mma"):
        q, sf, s = nvq.nvfp4_quantize_per_token(_dev(bits), sf_layout=layout)
        torch.cuda.synchronize()
        assert np.array_equal(_np(s).view(np.uint32), s_ref.view(np.uint32))
        assert np.array_equal(_np(q), q_ref)
        want = sf_ref if layout == "canonical" else oracle.sf_to_mma_layout(sf_ref)
        assert np.array_equal(_np(sf).reshape(want.shape), want)


@pytest.mark.parametrize("k", [-149, -140, -127, -120, -100, -91, -89])
def test_nvfp4_tiny_token_scales(nvq, k):
    # tokens whose coarse scale is subnormal or just around the fp32 fast-path threshold
    rng = np.random.default_rng(-k)
    x = rng.standard_normal((64, 256)) * 2688.0 * 2.0 ** k
    bits = _bits_of(x)
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(bits)
    q, sf, s = nvq.nvfp4_quantize_per_token(_dev(bits), sf_layout="canonical")
    assert np.array_equal(_np(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(_np(q), q_ref)
    assert np.array_equal(_np(sf).reshape(sf_ref.shape), sf_ref)


@pytest.mark.parametrize("K", [768, 1024, 2048])
@pytest.mark.parametrize("layout", ["canonical", "mma"])
def test_nvfp4_rows_on_different_paths(nvq, K, layout):
    """Rows of one warp whose coarse scales send them down different decision paths (tiny scales
    take the exact path, others the table path, zero rows have no scale): rows of at most 1024
    elements are quantized two to a warp, so neighbouring rows mix paths inside one warp."""
    rng = np.random.default_rng(K)
    R = 77                                          # odd: the last warp's second row is past the end
    x = rng.standard_normal((R, K)) * np.exp(rng.uniform(-3, 3, (R, 1)))
    kind = rng.integers(0, 4, R)
    x[kind == 1] *= 2688.0 * 2.0 ** -120            # exact path
    x[kind == 2] = 0.0                              # zero row
    bits = _bits_of(x)
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(bits)
    q, sf, s = nvq.nvfp4_quantize_per_token(_dev(bits), sf_layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(_np(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(_np(q), q_ref)
    if layout == "canonical":
        assert np.array_equal(_np(sf).reshape(sf_ref.shape), sf_ref)
    else:
        assert np.array_equal(_np(sf), oracle.sf_to_mma_layout(sf_ref))


def test_nvfp4_per_token_invariance_on_gpu(nvq):
    # a token's bytes do not depend on the rest of the batch (the scope the pages require)
    bits = family("random", (512, 768), seed=9)
    q, sf, s = nvq.nvfp4_quantize_per_token(_dev(bits), sf_layout="canonical")
    perm = np.random.default_rng(1).permutation(512)[:100]
    q2, sf2, s2 = nvq.nvfp4_quantize_per_token(_dev(np.ascontiguousarray(bits[perm])), sf_layout="canonical")
    assert torch.equal(q2, q[torch.from_numpy(perm).cuda()])
    assert torch.equal(s2, s[torch.from_numpy(perm).cuda()])


# ------------------------------------------------------------------------------------------------
# NVFP4 weights
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(3, 256, 192), (2, 80, 72), (1, 512, 384), (4, 64, 128), (2, 96, 136),
                                   (3, 48, 40), (1, 2080, 264)])
@pytest.mark.parametrize("layout", ["canonical", "mma"])
def test_nvfp4_weights_bit_exact(nvq, shape, layout):
    E, K, N = shape
    rng = np.random.default_rng(E * K + N)
    w = rng.standard_normal(shape) * 0.02 * np.exp(rng.uniform(-3, 3, (E, 1, 1)))
    w[0, :, : N // 2] *= 30.0                      # gate half larger than up half for expert 0
    bits = _bits_of(w)
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_weights(bits)
    q, sf, s = nvq.nvfp4_quantize_weights(_dev(bits).contiguous(), sf_layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(_np(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(_np(q), q_ref)
    if layout == "canonical":
        assert np.array_equal(_np(sf).reshape(sf_ref.shape), sf_ref)
    else:
        assert np.array_equal(_np(sf), oracle.sf_to_mma_layout(sf_ref.reshape(E * N, K // 16)))


@pytest.mark.parametrize("layout", ["canonical", "mma"])
def test_nvfp4_weights_tile_ranges_cross_experts(nvq, layout):
    """More 64 x 64 tiles (64 experts x 8 x 4) than encode CTAs, so each CTA's range of tiles
    crosses expert boundaries; three experts have a tiny coarse scale (exact decisions) between
    experts on the table-driven path."""
    E, K, N = 64, 512, 256
    rng = np.random.default_rng(7)
    w = rng.standard_normal((E, K, N)) * 0.02 * np.exp(rng.uniform(-2, 2, (E, 1, 1)))
    w[5:8] *= 2.0 ** -100
    bits = _bits_of(w)
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_weights(bits)
    assert (s_ref[5:8] < 2.0 ** -90).all() and (s_ref[8:] > 2.0 ** -90).all()
    q, sf, s = nvq.nvfp4_quantize_weights(_dev(bits).contiguous(), sf_layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(_np(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(_np(q), q_ref)
    if layout == "canonical":
        assert np.array_equal(_np(sf).reshape(sf_ref.shape), sf_ref)
    else:
        assert np.array_equal(_np(sf), oracle.sf_to_mma_layout(sf_ref.reshape(E * N, K // 16)))


@pytest.mark.parametrize("layout", ["canonical", "mma"])
def test_nvfp4_weights_product_and_boundary_scopes(nvq, layout):
    """Experts whose coarse scale is a power of two (s = 2^k: ties on the boundaries that no fp32
    multiplier reproduces, so the boundary comparison) next to experts with generic scales (the
    product path), in one launch; values on and next to the rounding midpoints."""
    E, K, N = 12, 256, 192
    bits = family("boundary", (E * K, N), seed=21).reshape(E, K, N)
    rng = np.random.default_rng(21)
    w = oracle.bf16_bits_to_f64(bits)
    w /= np.abs(w).reshape(E, -1).max(axis=1)[:, None, None]
    for e in range(E):
        k = int(rng.integers(-12, 4))
        amax = 2688.0 * 2.0 ** k if e % 2 == 0 else 2688.0 * 2.0 ** k * 1.37
        w[e] *= 0.5 * amax
        w[e, 0, 0] = amax
    bits = _bits_of(w)
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_weights(bits)
    assert (s_ref[0::2] == np.exp2(np.round(np.log2(s_ref[0::2])))).all()
    q, sf, s = nvq.nvfp4_quantize_weights(_dev(bits).contiguous(), sf_layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(_np(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(_np(q), q_ref)
    if layout == "canonical":
        assert np.array_equal(_np(sf).reshape(sf_ref.shape), sf_ref)
    else:
        assert np.array_equal(_np(sf), oracle.sf_to_mma_layout(sf_ref.reshape(E * N, K // 16)))


@pytest.mark.parametrize("layer", ["gate_up", "down"])
def test_full_size_expert_weights_sampled(nvq, layer):
    """All 128 expert matrices of the MoE layer in the bench's launch (MMA layout): every expert's
    scale, and 64 sampled output columns of 12 experts byte for byte."""
    K, N = (workloads.HIDDEN, 2 * workloads.INTERMEDIATE) if layer == "gate_up" else \
        (workloads.INTERMEDIATE, workloads.HIDDEN)
    w = workloads.expert_weights(K, N, seed=3, device="cuda")
    E = w.shape[0]
    q, sf, s = nvq.nvfp4_quantize_weights(w)
    torch.cuda.synchronize()
    amax = w.abs().reshape(E, -1).max(dim=1).values.float().cpu().numpy().astype(np.float64)
    s_ref = oracle.nvfp4_token_scale(amax)
    assert np.array_equal(_np(s).view(np.uint32), s_ref.view(np.uint32))
    rng = np.random.default_rng(11)
    kb = K // 16
    for e in rng.choice(E, 12, replace=False):
        cols = np.sort(rng.choice(N, 64, replace=False))
        we = oracle.bf16_bits_to_f64(workloads.to_bits(w[int(e)]))
        q_r, sf_r = oracle.nvfp4_quantize_rows(np.ascontiguousarray(we[:, cols].T), np.full(64, s_ref[e]))
        assert np.array_equal(_np(q[int(e)])[cols], q_r)
        r_idx, c_idx = np.meshgrid(int(e) * N + cols, np.arange(kb), indexing="ij")
        assert np.array_equal(_np(sf)[oracle.mma_layout_offset(r_idx, c_idx, kb)], sf_r)


# ------------------------------------------------------------------------------------------------
# Dequantize
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("fam", FAMILIES)
@pytest.mark.parametrize("layout", ["canonical", "mma"])
@pytest.mark.parametrize("out_offset", [0, 8])   # 8 bf16 = 16 bytes: output off the 32-byte grid
def test_dequantize_mxfp8_bit_exact(nvq, fam, layout, out_offset):
    bits = family(fam, (160, 224), seed=5)
    ref = oracle.mxfp8_quantize(bits, colwise=False)
    want = oracle.dequantize_mxfp8(ref["q_row"], ref["sf_row"])
    sf = ref["sf_row"] if layout == "canonical" else oracle.sf_to_mma_layout(ref["sf_row"])
    buf = torch.empty(160 * 224 + 16, dtype=torch.bfloat16, device="cuda")
    out = buf[out_offset:out_offset + 160 * 224].view(160, 224)
    nvq.dequantize_bf16(nvq.MXFP8, torch.from_numpy(ref["q_row"]).cuda(), torch.from_numpy(sf).cuda(),
                        rows=160, cols=224, sf_layout=layout, out=out)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fam", FAMILIES + ["tiny"])
@pytest.mark.parametrize("layout", ["canonical", "mma"])
@pytest.mark.parametrize("shape", [(96, 272), (100, 512)])     # two-block path; four-block path
def test_dequantize_nvfp4_rows_bit_exact(nvq, fam, layout, shape):
    R, C = shape
    if fam == "tiny":
        x = np.random.default_rng(6).standard_normal(shape) * 2.0 ** -120
        bits = _bits_of(x)
    else:
        bits = family(fam, shape, seed=6)
    q, sf, s = oracle.nvfp4_quantize_per_token(bits)
    want = oracle.dequantize_nvfp4(q, sf, s)
    sfl = sf if layout == "canonical" else oracle.sf_to_mma_layout(sf)
    out = nvq.dequantize_bf16(nvq.NVFP4, torch.from_numpy(q).cuda(), torch.from_numpy(sfl).cuda(),
                              torch.from_numpy(s).cuda(), nvq.SCOPE_ROW, rows=R, cols=C, sf_layout=layout)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("layout", ["canonical", "mma"])
@pytest.mark.parametrize("out_offset", [0, 8])   # 8 bf16 = 16 bytes: output off the 32-byte grid
def test_dequantize_nvfp4_weights_matrix_scope(nvq, layout, out_offset):
    # K = 128: rows of a multiple of 64 elements take the four-block path when the output is
    # 32-byte aligned and the two-block path otherwise; both give the oracle's bits
    E, K, N = 3, 128, 64
    rng = np.random.default_rng(7)
    bits = _bits_of(rng.standard_normal((E, K, N)) * 0.02)
    q, sf, s_w = oracle.nvfp4_quantize_weights(bits)
    sf2 = sf.reshape(E * N, K // 16)
    want = oracle.dequantize_nvfp4(q.reshape(E * N, K // 2), sf2, np.repeat(s_w, N))
    sfl = sf2 if layout == "canonical" else oracle.sf_to_mma_layout(sf2)
    buf = torch.empty(E * N * K + 16, dtype=torch.bfloat16, device="cuda")
    out = buf[out_offset:out_offset + E * N * K].view(E * N, K)
    nvq.dequantize_bf16(nvq.NVFP4, torch.from_numpy(q).cuda(), torch.from_numpy(sfl).cuda(),
                        torch.from_numpy(s_w).cuda(), nvq.SCOPE_MATRIX, groups=E, rows=N, cols=K,
                        sf_layout=layout, out=out)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)


# ------------------------------------------------------------------------------------------------
# Full-size workloads, sampled against the oracle
# ------------------------------------------------------------------------------------------------
def test_full_size_moe_activation_quant_sampled(nvq):
    counts, offsets = workloads.moe_routing()
    x = workloads.routed_activations(counts, offsets, workloads.HIDDEN, seed=11, device="cuda")
    q, sf, s = nvq.nvfp4_quantize_per_token(x, sf_layout="mma")
    mx = nvq.mxfp8_quantize(x, sf_layout="mma")
    torch.cuda.synchronize()
    R = x.shape[0]
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(R, 384, replace=False))
    xb = workloads.to_bits(x[torch.from_numpy(rows).cuda()])
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(xb)
    assert np.array_equal(_np(q[torch.from_numpy(rows).cuda()]), q_ref)
    assert np.array_equal(_np(s[torch.from_numpy(rows).cuda()]).view(np.uint32), s_ref.view(np.uint32))
    sf_all = _np(sf)
    kb = workloads.HIDDEN // 16
    r_idx, c_idx = np.meshgrid(rows, np.arange(kb), indexing="ij")
    assert np.array_equal(sf_all[oracle.mma_layout_offset(r_idx, c_idx, kb)], sf_ref)
    # MXFP8 rowwise on the same rows; columnwise on sampled 32-row bands
    mref = oracle.mxfp8_quantize(xb, colwise=False)
    assert np.array_equal(_np(mx["q_row"][torch.from_numpy(rows).cuda()]), mref["q_row"])
    bands = rng.choice(R // 32, 24, replace=False)
    for b in bands:
        xb2 = workloads.to_bits(x[32 * b:32 * b + 32])
        cref = oracle.mxfp8_quantize(xb2, rowwise=False)
        assert np.array_equal(_np(mx["q_colT"][:, 32 * b:32 * b + 32]), cref["q_colT"])
