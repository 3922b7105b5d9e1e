"""GPU parity of the scale-layout permutation and of the quantize-once gather against the oracle.

Scale layout [Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本", section
"重构权重更新接口": backend layouts explicit and verifiable]; gather [Miles-zh, section "逐 Token 激活值
缩放": one FP32 scale per token, so quantized tokens can be gathered instead of re-quantized].
"""
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


def _np(t):
    return t.detach().cpu().numpy()


def _tokens(T, K, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K)) * np.exp(rng.uniform(-6, 6, (T, 1)))
    x[rng.random((T, K)) < 0.05] = 0.0
    return oracle.f64_to_bf16_bits_rne(x)


@pytest.mark.parametrize("rows,kb", [(300, 7), (128, 4), (1, 1), (257, 130), (40, 128)])
def test_sf_layout_convert_both_ways(nvq, rows, kb):
    rng = np.random.default_rng(rows * 1000 + kb)
    sf = rng.integers(0, 256, (rows, kb), dtype=np.uint8)
    src = torch.from_numpy(sf.reshape(-1).copy()).cuda()
    mma = nvq.sf_layout_convert(src, rows, kb, "canonical", "mma")
    torch.cuda.synchronize()
    assert np.array_equal(_np(mma), oracle.sf_to_mma_layout(sf))
    back = nvq.sf_layout_convert(mma, rows, kb, "mma", "canonical")
    torch.cuda.synchronize()
    assert np.array_equal(_np(back).reshape(rows, kb), sf)
    assert np.array_equal(oracle.sf_from_mma_layout(_np(mma), rows, kb), sf)


def _index(T, rows, seed):
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, T, rows).astype(np.int32)
    idx[rng.random(rows) < 0.1] = -1                    # padding rows
    return idx


@pytest.mark.parametrize("src_layout,dst_layout", [("canonical", "canonical"), ("canonical", "mma"),
                                                   ("mma", "canonical"), ("mma", "mma")])
def test_gather_nvfp4_equals_oracle_and_requantization(nvq, src_layout, dst_layout):
    T, K, R = 200, 272, 333
    bits = _tokens(T, K, 5)
    idx = _index(T, R, 6)
    q, sf, s = nvq.nvfp4_quantize_per_token(workloads.from_bits(bits, "cuda"), sf_layout=src_layout)
    qg, sfg, sg = nvq.quantized_gather_rows(nvq.NVFP4, q, sf, s, torch.from_numpy(idx).cuda(), K,
                                            src_layout=src_layout, dst_layout=dst_layout)
    torch.cuda.synchronize()
    # oracle: quantize the tokens, then take rows (zero rows where idx = -1)
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(bits)
    keep = idx >= 0
    qe = np.zeros((R, K // 2), np.uint8); qe[keep] = q_ref[idx[keep]]
    sfe = np.zeros((R, K // 16), np.uint8); sfe[keep] = sf_ref[idx[keep]]
    se = np.zeros(R, np.float32); se[keep] = s_ref[idx[keep]]
    assert np.array_equal(_np(qg), qe)
    assert np.array_equal(_np(sg).view(np.uint32), se.view(np.uint32))
    sfe_l = sfe.reshape(-1) if dst_layout == "canonical" else oracle.sf_to_mma_layout(sfe)
    assert np.array_equal(_np(sfg).reshape(-1), sfe_l)
    # per-token invariance: the same bytes as quantizing the gathered bf16 rows
    xg = np.zeros((R, K), np.uint16); xg[keep] = bits[idx[keep]]
    q2, sf2, s2 = nvq.nvfp4_quantize_per_token(workloads.from_bits(xg, "cuda"), sf_layout=dst_layout)
    torch.cuda.synchronize()
    assert torch.equal(q2, qg) and torch.equal(sf2, sfg) and torch.equal(s2, sg)


def test_gather_mxfp8_rowwise_equals_oracle(nvq):
    T, K, R = 150, 320, 260
    bits = _tokens(T, K, 8)
    idx = _index(T, R, 9)
    o = nvq.mxfp8_quantize(workloads.from_bits(bits, "cuda"), colwise=False, sf_layout="mma")
    qg, sfg, sg = nvq.quantized_gather_rows(nvq.MXFP8, o["q_row"], o["sf_row"], None, torch.from_numpy(idx).cuda(),
                                            K, src_layout="mma", dst_layout="mma")
    torch.cuda.synchronize()
    assert sg is None
    ref = oracle.mxfp8_quantize(bits, colwise=False)
    keep = idx >= 0
    qe = np.zeros((R, K), np.uint8); qe[keep] = ref["q_row"][idx[keep]]
    sfe = np.zeros((R, K // 32), np.uint8); sfe[keep] = ref["sf_row"][idx[keep]]
    assert np.array_equal(_np(qg), qe)
    assert np.array_equal(_np(sfg), oracle.sf_to_mma_layout(sfe))


def test_gather_bad_index_sets_status_and_writes_zero_row(nvq):
    T, K = 16, 64
    bits = _tokens(T, K, 3)
    q, sf, s = nvq.nvfp4_quantize_per_token(workloads.from_bits(bits, "cuda"), sf_layout="canonical")
    idx = torch.tensor([0, 5, 16, -2, 3], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg, sfg, sg = nvq.quantized_gather_rows(nvq.NVFP4, q, sf, s, idx, K, src_layout="canonical",
                                            dst_layout="canonical", status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == nvq.DEV_BAD_INDEX
    assert torch.equal(qg[[0, 1, 4]], q[[0, 5, 3]])
    assert int(qg[2:4].abs().sum()) == 0 and float(sg[2:4].abs().sum()) == 0.0
    assert int(sfg.view(5, K // 16)[2:4].sum()) == 0


@pytest.mark.parametrize("align", [1, 32])
def test_full_size_quantize_once_dispatch(nvq, align):
    """16384 tokens x 2048, top-8 of 128 experts (Zipf 1.1), segments unpadded (the MoE bench step's
    layout) or padded to 32 rows: gathering the quantized tokens equals quantizing the gathered rows,
    byte for byte (the whole batch), and sampled rows equal the oracle."""
    T, K = 16384, workloads.HIDDEN
    choices = workloads.route_choices(T)
    counts = np.bincount(choices.reshape(-1), minlength=workloads.EXPERTS)
    offs = workloads.padded_offsets(counts, align)
    idx = workloads.dispatch_index(choices, offs)
    x = workloads.normal_bf16((T, K), 1.0, seed=21, device="cuda")
    q, sf, s = nvq.nvfp4_quantize_per_token(x)
    idx_d = torch.from_numpy(idx).cuda()
    qg, sfg, sg = nvq.quantized_gather_rows(nvq.NVFP4, q, sf, s, idx_d, K)
    xr = torch.zeros((idx.size, K), dtype=torch.bfloat16, device="cuda")
    keep = torch.from_numpy(idx >= 0).cuda()
    xr[keep] = x[idx_d[keep].long()]
    q2, sf2, s2 = nvq.nvfp4_quantize_per_token(xr)
    torch.cuda.synchronize()
    assert torch.equal(q2, qg) and torch.equal(sf2, sfg) and torch.equal(s2, sg)
    rows = np.random.default_rng(4).choice(np.flatnonzero(idx >= 0), 64, replace=False)
    tb = workloads.to_bits(x[torch.from_numpy(idx[rows]).long().cuda()].cpu())
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(tb)
    assert np.array_equal(_np(qg[torch.from_numpy(rows).cuda()]), q_ref)
    assert np.array_equal(_np(sg[torch.from_numpy(rows).cuda()]).view(np.uint32), s_ref.view(np.uint32))
    sf_rows = oracle.sf_from_mma_layout(_np(sfg), idx.size, K // 16)[rows]
    assert np.array_equal(sf_rows, sf_ref)
