"""GPU parity: the tcgen05 block-scaled grouped GEMM against the float64 oracle.

Inputs are quantized independently on both sides (GPU kernels vs oracle) from the same seeded bf16
data; the oracle multiplies its own dequantized operands in float64. Bound (method statement):
|D_gpu - D| <= 2e-3 * sum_k |s_a s_b deq(A) deq(B)|, checked on the fp32 output; the bf16 output
adds its own final rounding (at most 2^-8 |D|, half a bf16 ulp).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def nvq():
    import nvfp4_quantization_block_gb300 as m
    return m


def _bits(x):
    return oracle.f64_to_bf16_bits_rne(np.asarray(x, dtype=np.float64))


def _check(d_gpu, D, bound, bf16_out):
    d = d_gpu.detach().float().cpu().numpy().astype(np.float64)
    err = np.abs(d - D)
    allow = TOL * bound + (np.abs(D) * 2.0 ** -8 if bf16_out else 0.0)
    bad = err > allow
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside tolerance; worst err/bound "
                           f"{(err / np.maximum(bound, 1e-300)).max():.3e}")


def _routed(counts, k, seed, scale_rows=True, align=32):
    offs = workloads.padded_offsets(counts, align)
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((int(offs[-1]), k))
    if scale_rows:
        x *= np.exp(rng.uniform(-4, 4, (x.shape[0], 1)))
    x[~workloads.valid_row_mask(counts, offs)] = 0
    return offs, _bits(x)


# ------------------------------------------------------------------------------------------------
# forward / data-gradient (rows grouped by expert)
# ------------------------------------------------------------------------------------------------
def _run_m(nvq, fmt, counts, K, N, seed, out_type, align=32, offsets=None):
    E = len(counts)
    offs, xb = _routed(counts, K, seed, align=align)
    if offsets is not None:                       # explicit offsets (rows between groups are zero)
        offs = np.asarray(offsets, dtype=np.int64)
        xb = np.zeros((int(offs[-1]), K), dtype=np.uint16)
        rng0 = np.random.default_rng(seed)
        for e, c in enumerate(counts):
            xb[offs[e]:offs[e] + c] = _bits(rng0.standard_normal((c, K)) * np.exp(rng0.uniform(-4, 4, (c, 1))))
    rng = np.random.default_rng(seed + 1)
    wb = _bits(rng.standard_normal((E, K, N)) * 0.02 * np.exp(rng.uniform(-2, 2, (E, 1, 1))))
    x = workloads.from_bits(xb, "cuda")
    w = workloads.from_bits(wb, "cuda")
    M = x.shape[0]
    offs_d = torch.from_numpy(offs).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if fmt == "nvfp4":
        qa, sfa, sa = nvq.nvfp4_quantize_per_token(x, sf_layout="mma")
        qb, sfb, sb = nvq.nvfp4_quantize_weights(w.contiguous(), sf_layout="mma")
        d = nvq.block_scaled_grouped_gemm(nvq.NVFP4, nvq.GEMM_GROUP_M, qa, sfa, qb, sfb, offs_d, m=M, n=N, k=K,
                                          groups=E, s_a=sa, s_b=sb, out_type=out_type, status=status)
        qa_r, sfa_r, sa_r = oracle.nvfp4_quantize_per_token(xb)
        qb_r, sfb_r, sb_r = oracle.nvfp4_quantize_weights(wb)
        a = oracle.deq_operand("nvfp4", qa_r, sfa_r)
        b = np.stack([oracle.deq_operand("nvfp4", qb_r[e], sfb_r[e]) for e in range(E)])
        D, bound = oracle.grouped_gemm_reference("m", a, b, offs, sa_r, sb_r)
    else:
        # forward: A = rowwise MXFP8 of X; B[e] = columnwise MXFP8 of W[e] (blocks along K), i.e. W[e]^T
        qa = nvq.mxfp8_quantize(x, colwise=False, sf_layout="mma")
        wt = w.transpose(1, 2).contiguous().view(E * N, K)          # [E*N, K]: rows are W[e] columns
        qb = nvq.mxfp8_quantize(wt, colwise=False, sf_layout="mma")
        d = nvq.block_scaled_grouped_gemm(nvq.MXFP8, nvq.GEMM_GROUP_M, qa["q_row"], qa["sf_row"], qb["q_row"],
                                          qb["sf_row"], offs_d, m=M, n=N, k=K, groups=E, out_type=out_type,
                                          status=status)
        ra = oracle.mxfp8_quantize(xb, colwise=False)
        a = oracle.deq_operand("mxfp8", ra["q_row"], ra["sf_row"])
        b = []
        for e in range(E):
            rb = oracle.mxfp8_quantize(np.ascontiguousarray(wb[e]), rowwise=False)   # columnwise of W[e]
            b.append(oracle.deq_operand("mxfp8", rb["q_colT"], rb["sf_colT"]))
        D, bound = oracle.grouped_gemm_reference("m", a, np.stack(b), offs)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = ~np.isnan(D[:, 0])
    _check(d[torch.from_numpy(rows).cuda()], D[rows], bound[rows], out_type == nvq.OUT_BF16)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_contract_shape_single_group(nvq, fmt, out):
    # 256 x 512 by 512 x 384: one group, N not a multiple of the 256-column tile
    _run_m(nvq, fmt, [256], 512, 384, seed=0, out_type=nvq.OUT_F32 if out == "f32" else nvq.OUT_BF16)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("counts,K,N", [
    ([96, 0, 160, 33, 300], 256, 256),       # group starts at 32-row offsets inside scale tiles
    ([1, 31, 64, 0, 0, 129], 384, 512),      # K ragged against the FP4 stage (384 = 256 + 128)
    ([200, 77], 768, 384),
    ([0, 0, 0], 256, 256),                   # nothing to do
    ([40], 256, 256),                        # a single small group
    ([300, 40], 512, 256),                   # the last tile starts inside a scale tile
])
def test_grouped_rows(nvq, fmt, counts, K, N):
    _run_m(nvq, fmt, counts, K, N, seed=sum(counts) + K, out_type=nvq.OUT_F32)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("counts,K,N", [
    ([1, 16, 33, 250], 256, 256),            # group offsets 0, 1, 17, 50, 300: any row
    ([300, 41, 263, 97, 133], 512, 384),     # groups fill their tiles: bf16 box stores with ragged ends
    ([1, 31, 64, 0, 0, 129, 7], 384, 512),   # single rows, empty groups, K ragged against the FP4 stage
    ([127, 129, 255, 1, 128], 256, 256),     # every shift of a 128-row scale tile boundary nearby
])
def test_grouped_rows_any_offset(nvq, fmt, out, counts, K, N):
    _run_m(nvq, fmt, counts, K, N, seed=sum(counts) + K + 1, out_type=nvq.OUT_F32 if out == "f32" else nvq.OUT_BF16,
           align=1)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("counts,K,N", [
    ([16, 9, 25, 0, 17, 130, 1, 40], 512, 384),    # a group of more than 128 rows: two row tiles
    ([1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12], 384, 256),
    ([33] * 20, 1024, 640),                        # many tiles per CTA, 33 rows each (MMA N = 48)
])
def test_few_rows_per_group(nvq, fmt, out, counts, K, N):
    # decode-like groups (at most 64 rows on average, one of them over 128), unpadded offsets that
    # start anywhere inside the scale tiles
    assert sum(counts) <= 64 * len(counts)
    _run_m(nvq, fmt, counts, K, N, seed=sum(counts) + K + 3, out_type=nvq.OUT_F32 if out == "f32" else nvq.OUT_BF16,
           align=1)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_explicit_offsets_with_gaps(nvq, fmt):
    # offsets [0, 1, 17, 50, 300] with fewer real rows than each segment holds (rows between the
    # groups' rows are zero and belong to the groups), then a second call with gaps left out
    _run_m(nvq, fmt, [1, 16, 33, 250], 256, 256, seed=90, out_type=nvq.OUT_BF16, offsets=[0, 1, 17, 50, 300])
    _run_m(nvq, fmt, [1, 10, 20, 100], 256, 256, seed=91, out_type=nvq.OUT_F32, offsets=[0, 1, 17, 50, 300])


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("align", [32, 1])
def test_many_tiles_per_cta(nvq, fmt, align):
    # More tiles than CTAs: each CTA runs several tiles, so every stage ring wraps repeatedly, with
    # tiles starting inside a scale tile (32-row group offsets) mixed among aligned ones, and the
    # scale ring runs ahead of the operand ring across tile boundaries.
    counts = [150, 33, 260, 0, 121, 97, 201, 64, 180, 5, 140, 230]
    E, K, N = len(counts), 1024, 2560
    offs, xb = _routed(counts, K, seed=21, align=align)
    rng = np.random.default_rng(22)
    wb = _bits(rng.standard_normal((E, K, N)) * 0.02 * np.exp(rng.uniform(-2, 2, (E, 1, 1))))
    x = workloads.from_bits(xb, "cuda")
    w = workloads.from_bits(wb, "cuda")
    M = x.shape[0]
    offs_d = torch.from_numpy(offs).cuda()
    tiles_128 = sum(-(-int(r) // 128) for r in np.diff(offs)) * (N // 256)
    assert tiles_128 > 152                      # more tiles than a GB300 has SMs
    if fmt == "nvfp4":
        qa, sfa, sa = nvq.nvfp4_quantize_per_token(x)
        qb, sfb, sb = nvq.nvfp4_quantize_weights(w.contiguous())
        args, kw = (nvq.NVFP4, nvq.GEMM_GROUP_M, qa, sfa, qb, sfb, offs_d), dict(s_a=sa, s_b=sb)
        qa_r, sfa_r, sa_r = oracle.nvfp4_quantize_per_token(xb)
        qb_r, sfb_r, sb_r = oracle.nvfp4_quantize_weights(wb)
        a = oracle.deq_operand("nvfp4", qa_r, sfa_r)
        b = np.stack([oracle.deq_operand("nvfp4", qb_r[e], sfb_r[e]) for e in range(E)])
        D, bound = oracle.grouped_gemm_reference("m", a, b, offs, sa_r, sb_r)
    else:
        qa = nvq.mxfp8_quantize(x, colwise=False)
        qb = nvq.mxfp8_quantize(w.transpose(1, 2).contiguous().view(E * N, K), colwise=False)
        args, kw = (nvq.MXFP8, nvq.GEMM_GROUP_M, qa["q_row"], qa["sf_row"], qb["q_row"], qb["sf_row"], offs_d), {}
        ra = oracle.mxfp8_quantize(xb, colwise=False)
        a = oracle.deq_operand("mxfp8", ra["q_row"], ra["sf_row"])
        b = np.stack([oracle.deq_operand("mxfp8", *oracle.mxfp8_quantize(np.ascontiguousarray(wb[e]),
                                                                          rowwise=False).values())
                      for e in range(E)])
        D, bound = oracle.grouped_gemm_reference("m", a, b, offs)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = nvq.block_scaled_grouped_gemm(*args, m=M, n=N, k=K, groups=E, out_type=nvq.OUT_F32, status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _check(d, D, bound, False)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_box_store_epilogue_edges(nvq, fmt):
    """bf16 output of a grouped GEMM whose groups fill their row tiles (the epilogue's staged box
    stores): N = 384 (the last 256-column tile half full), an output view with a row pitch wider
    than N, and buffer rows after the last group; padding columns and those rows stay untouched."""
    counts = [300, 40, 0, 260, 97]
    E, K, N = len(counts), 512, 384
    offs, xb = _routed(counts, K, seed=41)
    extra = 64
    xb = np.concatenate([xb, np.zeros((extra, K), dtype=xb.dtype)])
    M = xb.shape[0]
    assert offs[-1] >= 128 * E                      # groups fill their tiles: box stores are used
    rng = np.random.default_rng(42)
    wb = _bits(rng.standard_normal((E, K, N)) * 0.02 * np.exp(rng.uniform(-2, 2, (E, 1, 1))))
    x = workloads.from_bits(xb, "cuda")
    w = workloads.from_bits(wb, "cuda")
    offs_d = torch.from_numpy(offs).cuda()
    big = torch.full((M, N + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    d = big[:, :N]
    if fmt == "nvfp4":
        qa, sfa, sa = nvq.nvfp4_quantize_per_token(x)
        qb, sfb, sb = nvq.nvfp4_quantize_weights(w.contiguous())
        nvq.block_scaled_grouped_gemm(nvq.NVFP4, nvq.GEMM_GROUP_M, qa, sfa, qb, sfb, offs_d, m=M, n=N, k=K, groups=E,
                                      s_a=sa, s_b=sb, out=d)
        qa_r, sfa_r, sa_r = oracle.nvfp4_quantize_per_token(xb)
        qb_r, sfb_r, sb_r = oracle.nvfp4_quantize_weights(wb)
        a = oracle.deq_operand("nvfp4", qa_r, sfa_r)
        b = np.stack([oracle.deq_operand("nvfp4", qb_r[e], sfb_r[e]) for e in range(E)])
        D, bound = oracle.grouped_gemm_reference("m", a, b, offs, sa_r, sb_r)
    else:
        qa = nvq.mxfp8_quantize(x, colwise=False)
        qb = nvq.mxfp8_quantize(w.transpose(1, 2).contiguous().view(E * N, K), colwise=False)
        nvq.block_scaled_grouped_gemm(nvq.MXFP8, nvq.GEMM_GROUP_M, qa["q_row"], qa["sf_row"], qb["q_row"],
                                      qb["sf_row"], offs_d, m=M, n=N, k=K, groups=E, out=d)
        ra = oracle.mxfp8_quantize(xb, colwise=False)
        a = oracle.deq_operand("mxfp8", ra["q_row"], ra["sf_row"])
        b = np.stack([oracle.deq_operand("mxfp8", *oracle.mxfp8_quantize(np.ascontiguousarray(wb[e]),
                                                                          rowwise=False).values())
                      for e in range(E)])
        D, bound = oracle.grouped_gemm_reference("m", a, b, offs)
    torch.cuda.synchronize()
    rows = ~np.isnan(D[:, 0])
    assert rows.sum() == offs[-1]
    _check(d[torch.from_numpy(rows).cuda()], D[rows], bound[rows], True)
    host = big.float().cpu().numpy()
    assert (host[:, N:] == 7.0).all()               # columns past N
    assert (host[int(offs[-1]):, :] == 7.0).all()   # rows after the last group


def test_rows_outside_groups_untouched(nvq):
    E, K, N = 2, 256, 256
    counts = [40, 20]
    offs = np.array([0, 64, 96], dtype=np.int64)       # 96 of 160 buffer rows belong to groups
    rng = np.random.default_rng(3)
    xb = _bits(rng.standard_normal((160, K)))
    wb = _bits(rng.standard_normal((E, K, N)) * 0.02)
    x = workloads.from_bits(xb, "cuda")
    qa, sfa, sa = nvq.nvfp4_quantize_per_token(x, sf_layout="mma")
    qb, sfb, sb = nvq.nvfp4_quantize_weights(workloads.from_bits(wb, "cuda").contiguous(), sf_layout="mma")
    d = torch.full((160, N), 7.0, dtype=torch.float32, device="cuda")
    nvq.block_scaled_grouped_gemm(nvq.NVFP4, nvq.GEMM_GROUP_M, qa, sfa, qb, sfb, torch.from_numpy(offs).cuda(),
                                  m=160, n=N, k=K, groups=E, s_a=sa, s_b=sb, out=d, out_type=nvq.OUT_F32)
    torch.cuda.synchronize()
    assert torch.all(d[96:] == 7.0)
    assert not torch.all(d[:96] == 7.0)
    del counts


def test_bad_offsets_set_status_and_write_nothing(nvq):
    K, N = 256, 256
    x = workloads.normal_bf16((64, K), device="cuda")
    w = workloads.normal_bf16((2, K, N), 0.02, device="cuda")
    qa, sfa, sa = nvq.nvfp4_quantize_per_token(x, sf_layout="mma")
    qb, sfb, sb = nvq.nvfp4_quantize_weights(w, sf_layout="mma")
    d = torch.full((64, N), 3.0, dtype=torch.float32, device="cuda")
    for bad in ([0, 96, 64], [0, 32, 16], [16, 64, 64]):   # past the buffer / not monotone / [0] != 0
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        nvq.block_scaled_grouped_gemm(nvq.NVFP4, nvq.GEMM_GROUP_M, qa, sfa, qb, sfb,
                                      torch.tensor(bad, dtype=torch.int64, device="cuda"), m=64, n=N, k=K,
                                      groups=2, s_a=sa, s_b=sb, out=d, out_type=nvq.OUT_F32, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == nvq.DEV_BAD_OFFSETS
        assert torch.all(d == 3.0)
    # weight gradients: reduction offsets must be multiples of 32
    qx = nvq.mxfp8_quantize(workloads.normal_bf16((64, 128), device="cuda"), rowwise=False)
    dk = torch.full((2, 128, 128), 3.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nvq.block_scaled_grouped_gemm(nvq.MXFP8, nvq.GEMM_GROUP_K, qx["q_colT"], qx["sf_colT"], qx["q_colT"],
                                  qx["sf_colT"], torch.tensor([0, 48, 64], dtype=torch.int64, device="cuda"),
                                  m=128, n=128, k=64, groups=2, out=dk, out_type=nvq.OUT_F32, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == nvq.DEV_BAD_OFFSETS
    assert torch.all(dk == 3.0)


def test_host_rejects_bad_shapes(nvq):
    x = torch.zeros((64, 256), dtype=torch.uint8, device="cuda")
    offs = torch.tensor([0, 64], dtype=torch.int64, device="cuda")
    with pytest.raises(nvq.NvqError):        # k not a multiple of 128
        nvq.block_scaled_grouped_gemm(nvq.MXFP8, nvq.GEMM_GROUP_M, x, x, x, x, offs, m=64, n=256, k=96, groups=1)
    with pytest.raises(nvq.NvqError):        # n not a multiple of 128
        nvq.block_scaled_grouped_gemm(nvq.MXFP8, nvq.GEMM_GROUP_M, x, x, x, x, offs, m=64, n=200, k=256, groups=1)
    with pytest.raises(nvq.NvqError):        # NVFP4 weight gradient is not part of the method
        nvq.block_scaled_grouped_gemm(nvq.NVFP4, nvq.GEMM_GROUP_K, x, x, x, x, offs, m=128, n=256, k=256, groups=1)


# ------------------------------------------------------------------------------------------------
# weight gradient (reduction grouped by expert), MXFP8 columnwise copies
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("counts,Kin,Nout", [([64, 0, 96, 200], 256, 256), ([33, 300], 128, 384),
                                             ([500, 40], 384, 256)])
def test_weight_gradient_grouped_k(nvq, counts, Kin, Nout):
    offs, xb = _routed(counts, Kin, seed=5)
    rng = np.random.default_rng(6)
    dy = rng.standard_normal((int(offs[-1]), Nout)) * 1e-3
    dy[~workloads.valid_row_mask(counts, offs)] = 0
    dyb = _bits(dy)
    x = workloads.from_bits(xb, "cuda")
    g = workloads.from_bits(dyb, "cuda")
    Mtot = x.shape[0]
    E = len(counts)
    qx = nvq.mxfp8_quantize(x, rowwise=False, sf_layout="mma")
    qg = nvq.mxfp8_quantize(g, rowwise=False, sf_layout="mma")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = nvq.block_scaled_grouped_gemm(nvq.MXFP8, nvq.GEMM_GROUP_K, qx["q_colT"], qx["sf_colT"], qg["q_colT"],
                                      qg["sf_colT"], torch.from_numpy(offs).cuda(), m=Kin, n=Nout, k=Mtot,
                                      groups=E, out_type=nvq.OUT_F32, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rx = oracle.mxfp8_quantize(xb, rowwise=False)
    rg = oracle.mxfp8_quantize(dyb, rowwise=False)
    A = oracle.deq_operand("mxfp8", rx["q_colT"], rx["sf_colT"])
    B = oracle.deq_operand("mxfp8", rg["q_colT"], rg["sf_colT"])
    D, bound = oracle.grouped_gemm_reference("k", A, B, offs)
    _check(d, D, bound, False)


# ------------------------------------------------------------------------------------------------
# Full-size workloads in the benchmark's launch configuration, sampled against the oracle
# ------------------------------------------------------------------------------------------------
def _sample_pairs(rng, rows, n, count):
    return rng.choice(rows, count), rng.integers(0, n, count)


def _oracle_weight_columns(w_e_bits, cols):
    """Oracle NVFP4 of selected output columns of one expert matrix W[e] [K, N] (bf16 bits): the
    expert's FP32 scale from the whole matrix's amax, then the columns' 1x16 blocks along K.
    Returns (dequantized rows [len(cols), K] without the FP32 scale, the FP32 scale)."""
    wf = oracle.bf16_bits_to_f64(w_e_bits)
    s_w = oracle.nvfp4_token_scale(np.abs(wf).max())
    q, sf = oracle.nvfp4_quantize_rows(np.ascontiguousarray(wf[:, cols].T), np.full(len(cols), s_w))
    return oracle.deq_operand("nvfp4", q, sf), float(s_w)


def test_full_size_dense_mxfp8_sampled(nvq):
    inp = workloads.dense_inputs(seed=0, device="cuda")
    x, w = inp["x"], inp["w"]
    M, K = x.shape
    N = w.shape[1]
    qa = nvq.mxfp8_quantize(x, colwise=False)
    qb = nvq.mxfp8_quantize(w, rowwise=False)          # columnwise of W: [N, K], blocks along K
    offs = torch.tensor([0, M], dtype=torch.int64, device="cuda")
    d = nvq.block_scaled_grouped_gemm(nvq.MXFP8, nvq.GEMM_GROUP_M, qa["q_row"], qa["sf_row"], qb["q_colT"],
                                      qb["sf_colT"], offs, m=M, n=N, k=K, groups=1)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    ii, jj = _sample_pairs(rng, M, N, 2048)
    xa = workloads.to_bits(x[torch.from_numpy(ii).cuda()])
    wc = workloads.to_bits(w[:, torch.from_numpy(jj).cuda()].T.contiguous())
    ra = oracle.mxfp8_quantize(xa, colwise=False)
    rb = oracle.mxfp8_quantize(wc, colwise=False)      # rows of W^T = columns of W, blocks along K
    A = oracle.deq_operand("mxfp8", ra["q_row"], ra["sf_row"])
    B = oracle.deq_operand("mxfp8", rb["q_row"], rb["sf_row"])
    Dv, bd = oracle.grouped_gemm_entries("m", A, B, np.tile([0, K], (len(ii), 1)), np.ones(len(ii)))
    got = d[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()]
    _check(got, Dv, bd, True)


@pytest.mark.parametrize("layer,align", [("gate_up", 1), ("gate_up", 32), ("down", 1)])
def test_full_size_moe_nvfp4_sampled(nvq, layer, align):
    # the bench's MoE layer (unpadded expert segments) and the 32-row padded layout: gate_up
    # (K = 2048, N = 1536) and down (K = 768, N = 2048) over the 131072 Zipf-routed rows
    counts, offs = workloads.moe_routing(align=align)
    K, N = (workloads.HIDDEN, 2 * workloads.INTERMEDIATE) if layer == "gate_up" else \
        (workloads.INTERMEDIATE, workloads.HIDDEN)
    x = workloads.routed_activations(counts, offs, K, seed=1, device="cuda")
    w = workloads.expert_weights(K, N, seed=2, device="cuda")
    qa, sfa, sa = nvq.nvfp4_quantize_per_token(x)
    qb, sfb, sb = nvq.nvfp4_quantize_weights(w)
    M, E = x.shape[0], w.shape[0]
    d = nvq.block_scaled_grouped_gemm(nvq.NVFP4, nvq.GEMM_GROUP_M, qa, sfa, qb, sfb, torch.from_numpy(offs).cuda(),
                                      m=M, n=N, k=K, groups=E, s_a=sa, s_b=sb)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    experts = np.concatenate([rng.choice(E, 6, replace=False), [int(np.argmax(counts)), int(np.argmin(counts))]])
    for e in experts:
        if counts[e] == 0:
            continue
        rows = offs[e] + rng.integers(0, counts[e], 64)
        cols = rng.integers(0, N, 64)
        xa = workloads.to_bits(x[torch.from_numpy(rows).cuda()])
        q_r, sf_r, s_r = oracle.nvfp4_quantize_per_token(xa)
        A = oracle.deq_operand("nvfp4", q_r, sf_r)
        B, s_w = _oracle_weight_columns(workloads.to_bits(w[int(e)]), cols)
        Dv, bd = oracle.grouped_gemm_entries("m", A, B, np.tile([0, K], (64, 1)), s_r.astype(np.float64) * s_w)
        got = d[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
        _check(got, Dv, bd, True)


@pytest.mark.parametrize("layer", ["gate_up", "down"])
def test_full_size_mxfp8_data_gradient_sampled(nvq, layer):
    # the backward workload's data gradients: dX = dY W[e]^T per expert, A = rowwise MXFP8 of dY
    # [R, N] (blocks along N), B = rowwise MXFP8 of W stacked [E*K, N] (W[e] [K, N])
    counts, offs = workloads.moe_routing()
    K, N = (workloads.HIDDEN, 2 * workloads.INTERMEDIATE) if layer == "gate_up" else \
        (workloads.INTERMEDIATE, workloads.HIDDEN)
    E = len(counts)
    g = workloads.routed_activations(counts, offs, N, std=1e-3, seed=5, device="cuda")
    w = workloads.expert_weights(K, N, seed=3, device="cuda").view(E * K, N)
    qg = nvq.mxfp8_quantize(g, colwise=False)
    qw = nvq.mxfp8_quantize(w, colwise=False)
    M = g.shape[0]
    d = nvq.block_scaled_grouped_gemm(nvq.MXFP8, nvq.GEMM_GROUP_M, qg["q_row"], qg["sf_row"], qw["q_row"],
                                      qw["sf_row"], torch.from_numpy(offs).cuda(), m=M, n=K, k=N, groups=E)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    for e in np.concatenate([rng.choice(E, 5, replace=False), [int(np.argmax(counts))]]):
        if counts[e] == 0:
            continue
        rows = offs[e] + rng.integers(0, counts[e], 64)
        cols = rng.integers(0, K, 64)
        ga = workloads.to_bits(g[torch.from_numpy(rows).cuda()])
        wr = workloads.to_bits(w[torch.from_numpy(int(e) * K + cols).cuda()])
        A = oracle.deq_operand("mxfp8", *oracle.mxfp8_quantize(ga, colwise=False).values())
        B = oracle.deq_operand("mxfp8", *oracle.mxfp8_quantize(wr, colwise=False).values())
        Dv, bd = oracle.grouped_gemm_entries("m", A, B, np.tile([0, N], (64, 1)), np.ones(64))
        got = d[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
        _check(got, Dv, bd, True)


@pytest.mark.parametrize("layer", ["gate_up", "down"])
def test_full_size_decode_nvfp4(nvq, layer):
    # the decode workload: 256 tokens, uniform top-8 over 128 experts (9..25 rows each, 2048 rows,
    # unpadded); gate_up K = 2048, N = 1536 or down K = 768, N = 2048; every row of 24 experts
    # checked on 96 columns
    counts = workloads.route_counts(256, zipf_s=0.0, seed=0)
    offs = workloads.padded_offsets(counts, 1)
    K, N = (workloads.HIDDEN, 2 * workloads.INTERMEDIATE) if layer == "gate_up" else \
        (workloads.INTERMEDIATE, workloads.HIDDEN)
    E = workloads.EXPERTS
    x = workloads.routed_activations(counts, offs, K, seed=1, device="cuda")
    w = workloads.expert_weights(K, N, seed=3 if layer == "gate_up" else 4, device="cuda")
    qa, sfa, sa = nvq.nvfp4_quantize_per_token(x)
    qb, sfb, sb = nvq.nvfp4_quantize_weights(w)
    M = x.shape[0]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = nvq.block_scaled_grouped_gemm(nvq.NVFP4, nvq.GEMM_GROUP_M, qa, sfa, qb, sfb, torch.from_numpy(offs).cuda(),
                                      m=M, n=N, k=K, groups=E, s_a=sa, s_b=sb, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and M == 2048
    q_r, sf_r, s_r = oracle.nvfp4_quantize_per_token(workloads.to_bits(x))
    A = oracle.deq_operand("nvfp4", q_r, sf_r)
    rng = np.random.default_rng(6)
    experts = np.concatenate([rng.choice(E, 22, replace=False), [int(np.argmax(counts)), int(np.argmin(counts))]])
    for e in experts:
        cols = rng.integers(0, N, 96)
        B, s_w = _oracle_weight_columns(workloads.to_bits(w[int(e)]), cols)
        rows = np.arange(offs[e], offs[e + 1])
        ii, jj = np.repeat(rows, 96), np.tile(np.arange(96), len(rows))
        Dv, bd = oracle.grouped_gemm_entries("m", A[ii], B[jj], np.tile([0, K], (len(ii), 1)),
                                             s_r[ii].astype(np.float64) * s_w)
        got = d[torch.from_numpy(ii).cuda(), torch.from_numpy(cols[jj]).cuda()]
        _check(got, Dv, bd, True)


def test_full_size_weight_gradient_sampled(nvq):
    counts, offs = workloads.moe_routing()
    Kin, Nout = workloads.HIDDEN, 2 * workloads.INTERMEDIATE
    x = workloads.routed_activations(counts, offs, Kin, seed=3, device="cuda")
    g = workloads.routed_activations(counts, offs, Nout, std=1e-3, seed=4, device="cuda")
    qx = nvq.mxfp8_quantize(x, rowwise=False)
    qg = nvq.mxfp8_quantize(g, rowwise=False)
    E = len(counts)
    d = nvq.block_scaled_grouped_gemm(nvq.MXFP8, nvq.GEMM_GROUP_K, qx["q_colT"], qx["sf_colT"], qg["q_colT"],
                                      qg["sf_colT"], torch.from_numpy(offs).cuda(), m=Kin, n=Nout, k=x.shape[0],
                                      groups=E)
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    S = 256
    ee = rng.integers(0, E, S)
    ii = rng.integers(0, Kin, S)
    jj = rng.integers(0, Nout, S)
    xa = workloads.to_bits(x[:, torch.from_numpy(ii).cuda()].T.contiguous())     # [S, Mtot] columns of X
    ga = workloads.to_bits(g[:, torch.from_numpy(jj).cuda()].T.contiguous())
    A = oracle.deq_operand("mxfp8", *oracle.mxfp8_quantize(xa, colwise=False).values())
    B = oracle.deq_operand("mxfp8", *oracle.mxfp8_quantize(ga, colwise=False).values())
    Dv, bd = oracle.grouped_gemm_entries("k", A, B, np.stack([offs[ee], offs[ee + 1]], 1), np.ones(S))
    got = d[torch.from_numpy(ee).cuda(), torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()]
    _check(got, Dv, bd, True)


# ------------------------------------------------------------------------------------------------
# BF16 grouped GEMM (high-precision and dequantized backward) [Miles-zh, "高精度反向和去量化反向"]
# ------------------------------------------------------------------------------------------------
def _bf16_m(nvq, counts, K, N, seed, out_type, align=32):
    E = len(counts)
    offs, xb = _routed(counts, K, seed, align=align)
    rng = np.random.default_rng(seed + 1)
    wb = _bits(rng.standard_normal((E, N, K)) * 0.02 * np.exp(rng.uniform(-2, 2, (E, 1, 1))))   # B[e] [N, K]
    x = workloads.from_bits(xb, "cuda")
    w = workloads.from_bits(wb, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = nvq.block_scaled_grouped_gemm(nvq.BF16, nvq.GEMM_GROUP_M, x, None, w, None, torch.from_numpy(offs).cuda(),
                                      m=x.shape[0], n=N, k=K, groups=E, out_type=out_type, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    D, bound = oracle.grouped_gemm_reference("m", oracle.bf16_bits_to_f64(xb), oracle.bf16_bits_to_f64(wb), offs)
    rows = ~np.isnan(D[:, 0])
    _check(d[torch.from_numpy(rows).cuda()], D[rows], bound[rows], out_type == nvq.OUT_BF16)


@pytest.mark.parametrize("counts,K,N,out", [
    ([256], 512, 384, "f32"),                    # one group, N ragged against the 256-column tile
    ([256], 512, 384, "bf16"),
    ([96, 0, 160, 33, 300], 256, 256, "f32"),    # group starts at 32-row offsets
    ([1, 31, 64, 0, 0, 129], 80, 512, "f32"),    # K ragged against the 64-element stage
    ([0, 0, 0], 256, 256, "f32"),
])
def test_bf16_grouped_rows(nvq, counts, K, N, out):
    _bf16_m(nvq, counts, K, N, seed=sum(counts) + K, out_type=nvq.OUT_F32 if out == "f32" else nvq.OUT_BF16)


def test_bf16_many_tiles_per_cta(nvq):
    # more tiles than CTAs: the stage ring wraps across tiles of different groups
    _bf16_m(nvq, [150, 33, 260, 0, 121, 97, 201, 64, 180, 5, 140, 230], 1024, 2560, seed=31, out_type=nvq.OUT_F32)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_bf16_few_rows_per_group(nvq, out):
    _bf16_m(nvq, [16, 9, 25, 0, 17, 130, 1, 40], 272, 384, seed=34,
            out_type=nvq.OUT_F32 if out == "f32" else nvq.OUT_BF16, align=1)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_bf16_any_offset(nvq, out):
    _bf16_m(nvq, [300, 41, 263, 97, 133, 1], 256, 384, seed=33,
            out_type=nvq.OUT_F32 if out == "f32" else nvq.OUT_BF16, align=1)


@pytest.mark.parametrize("counts,Kin,Nout", [([500, 40], 384, 256), ([100, 0, 250, 33], 256, 384)])
def test_bf16_weight_gradient_grouped_k(nvq, counts, Kin, Nout):
    # dW[e] = X_e^T dY_e with X^T [Kin, R] and dY^T [Nout, R] (K-major over the routed rows)
    offs, xb = _routed(counts, Kin, seed=7)
    rng = np.random.default_rng(8)
    dy = rng.standard_normal((int(offs[-1]), Nout)) * 1e-3
    dy[~workloads.valid_row_mask(counts, offs)] = 0
    xt, gt = np.ascontiguousarray(xb.T), np.ascontiguousarray(_bits(dy).T)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = nvq.block_scaled_grouped_gemm(nvq.BF16, nvq.GEMM_GROUP_K, workloads.from_bits(xt, "cuda"), None,
                                      workloads.from_bits(gt, "cuda"), None, torch.from_numpy(offs).cuda(),
                                      m=Kin, n=Nout, k=xt.shape[1], groups=len(counts), out_type=nvq.OUT_F32,
                                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    D, bound = oracle.grouped_gemm_reference("k", oracle.bf16_bits_to_f64(xt), oracle.bf16_bits_to_f64(gt), offs)
    _check(d, D, bound, False)


def test_bf16_dequantized_backward_dgrad(nvq):
    """Dequantized backward, data gradient: dX = dY W^T per expert with W the BF16 dequantization of
    its MXFP8 rowwise copy (blocks along the output dimension, the reduction dimension here)."""
    counts, Kin, Nout = [130, 0, 61, 200], 256, 384
    E = len(counts)
    offs, gb = _routed(counts, Nout, seed=12)
    rng = np.random.default_rng(13)
    wb = _bits(rng.standard_normal((E * Kin, Nout)) * 0.02)               # W[e] [Kin, Nout], stacked
    qw = nvq.mxfp8_quantize(workloads.from_bits(wb, "cuda"), colwise=False, sf_layout="mma")
    wdq = nvq.dequantize_bf16(nvq.MXFP8, qw["q_row"], qw["sf_row"], rows=E * Kin, cols=Nout)
    g = workloads.from_bits(gb, "cuda")
    d = nvq.block_scaled_grouped_gemm(nvq.BF16, nvq.GEMM_GROUP_M, g, None, wdq, None, torch.from_numpy(offs).cuda(),
                                      m=g.shape[0], n=Kin, k=Nout, groups=E, out_type=nvq.OUT_F32)
    torch.cuda.synchronize()
    rw = oracle.mxfp8_quantize(wb, colwise=False)
    wdq_ref = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits_rne(oracle.deq_operand("mxfp8", rw["q_row"], rw["sf_row"])))
    assert np.array_equal(workloads.to_bits(wdq.cpu()), oracle.f64_to_bf16_bits_rne(wdq_ref))   # the dequantization
    D, bound = oracle.grouped_gemm_reference("m", oracle.bf16_bits_to_f64(gb), wdq_ref.reshape(E, Kin, Nout), offs)
    rows = ~np.isnan(D[:, 0])
    _check(d[torch.from_numpy(rows).cuda()], D[rows], bound[rows], False)


# ------------------------------------------------------------------------------------------------
# the documented maximum of 1024 groups
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_max_groups(nvq, fmt):
    """1024 groups (the maximum), most of them empty, a few with rows at 32-row offsets: the tile
    schedule's group search and the device offset checks at full size."""
    counts = [0] * 1024
    for e, c in [(0, 40), (7, 32), (300, 96), (511, 1), (512, 33), (1000, 64), (1023, 130)]:
        counts[e] = c
    _run_m(nvq, fmt, counts, 128, 128, seed=77, out_type=nvq.OUT_F32)


def test_more_than_max_groups_is_rejected(nvq):
    x = torch.zeros((64, 128), dtype=torch.uint8, device="cuda")
    offs = torch.zeros(1026, dtype=torch.int64, device="cuda")
    with pytest.raises(nvq.NvqError):
        nvq.block_scaled_grouped_gemm(nvq.MXFP8, nvq.GEMM_GROUP_M, x, x, x, x, offs, m=64, n=128, k=128, groups=1025)
