"""GPU parity of the fused SwiGLU + per-token NVFP4 quantizer against the oracle, byte for byte.

[Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本", section "逐 Token 激活值
缩放": SwiGLU experts run gate and up as one fused GEMM; one call emits FP4 values, E4M3 block scales
and per-token FP32 scales.] The oracle computes the SwiGLU in the same float32 steps
(oracle/swiglu.py) and quantizes its bf16 result with its own per-token NVFP4.
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


def _gate_up(R, I, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((R, I)) * np.exp(rng.uniform(-3, 4, (R, 1)))
    u = rng.standard_normal((R, I)) * np.exp(rng.uniform(-3, 3, (R, 1)))
    g[rng.random((R, I)) < 0.01] *= 60.0          # gates with |g| > 87 scattered in every row
    g[rng.random((R, I)) < 0.02] = 0.0
    # rows whose gates make exp(-g) leave float32's range (-g in (87, 300] and beyond the clamp)
    # with up values large enough that silu(g) u stays a normal number
    wide = np.arange(R) % 7 == 3
    g[wide] = -rng.uniform(85.0, 110.0, (wide.sum(), I))
    g[wide & (np.arange(R) % 14 == 3)] *= rng.choice([1.0, 3.0, 1e36], (int((wide & (np.arange(R) % 14 == 3)).sum()), I))
    u[wide] = rng.standard_normal((wide.sum(), I)) * 10.0 ** rng.uniform(28, 38, (wide.sum(), 1))
    bits = oracle.f64_to_bf16_bits_rne(np.concatenate([g, u], axis=1))
    bits[:, :I][np.random.default_rng(seed + 1).random((R, I)) < 0.01] = 0x8000   # negative zero gates
    return bits


def _check(nvq, bits, layout, out):
    R, I = bits.shape[0], bits.shape[1] // 2
    q, sf, s = out
    h = oracle.swiglu_rows(bits)
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(h)
    assert np.array_equal(_np(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(_np(q), q_ref)
    if layout == "canonical":
        assert np.array_equal(_np(sf).reshape(sf_ref.shape), sf_ref)
    else:
        assert np.array_equal(_np(sf), oracle.sf_to_mma_layout(sf_ref))


@pytest.mark.parametrize("R,I", [(300, 768), (129, 48), (64, 272), (5, 2048 + 16)])
@pytest.mark.parametrize("layout", ["canonical", "mma"])
def test_swiglu_quantize_bit_exact(nvq, R, I, layout):
    bits = _gate_up(R, I, seed=R + I)
    out = nvq.nvfp4_swiglu_quantize_per_token(workloads.from_bits(bits, "cuda"), sf_layout=layout)
    torch.cuda.synchronize()
    _check(nvq, bits, layout, out)


def test_swiglu_quantize_many_row_groups_per_warp(nvq):
    # 13001 rows of 256 + 256: 6501 two-row groups, more than a 152-SM GPU holds resident warps, so
    # each warp takes two or three in turn and the last turn is ragged (moderate gates and up values:
    # over this many rows the extreme rows of _gate_up can overflow bf16)
    R, I = 13001, 256
    rng = np.random.default_rng(21)
    g = rng.standard_normal((R, I)) * np.exp(rng.uniform(-3, 4, (R, 1)))
    u = rng.standard_normal((R, I)) * np.exp(rng.uniform(-3, 3, (R, 1)))
    g[rng.random((R, I)) < 0.01] *= 60.0                  # gates with |g| > 87 in most rows
    bits = oracle.f64_to_bf16_bits_rne(np.concatenate([g, u], axis=1))
    for layout in ("canonical", "mma"):
        out = nvq.nvfp4_swiglu_quantize_per_token(workloads.from_bits(bits, "cuda"), sf_layout=layout)
        torch.cuda.synchronize()
        _check(nvq, bits, layout, out)


def test_swiglu_quantize_division_ranges(nvq):
    # the division g / (1 + exp(-g)) over the ranges its fast steps cover and those they leave to
    # IEEE division: quotients near 2^-100 (tiny gates, huge exp(-g)), subnormal and zero gates
    R, I = 64, 512
    rng = np.random.default_rng(17)
    g = rng.standard_normal((R, I))
    kind = np.arange(R) % 4
    g[kind == 0] = -rng.uniform(55.0, 87.0, ((kind == 0).sum(), I))          # exp(-g) up to 2^125
    g[kind == 1] = np.sign(rng.standard_normal(((kind == 1).sum(), I))) * 2.0 ** rng.uniform(-133, -90, ((kind == 1).sum(), I))
    g[kind == 2] *= 2.0 ** rng.integers(-110, 10, ((kind == 2).sum(), I))
    u = rng.standard_normal((R, I)) * 10.0 ** rng.uniform(-3, 35, (R, 1))
    bits = oracle.f64_to_bf16_bits_rne(np.concatenate([g, u], axis=1))
    bits[3, :I:7] = 0x8000                                                   # negative zero gates
    bits[3, 1:I:7] = 0x0000
    out = nvq.nvfp4_swiglu_quantize_per_token(workloads.from_bits(bits, "cuda"), sf_layout="canonical")
    torch.cuda.synchronize()
    _check(nvq, bits, "canonical", out)


def test_swiglu_quantize_strided_rows(nvq):
    R, I = 96, 256
    bits = _gate_up(R, I, seed=3)
    wide = np.zeros((R, 2 * I + 40), np.uint16)
    wide[:, :2 * I] = bits
    x = workloads.from_bits(wide, "cuda")[:, :2 * I]
    out = nvq.nvfp4_swiglu_quantize_per_token(x, sf_layout="mma")
    torch.cuda.synchronize()
    _check(nvq, bits, "mma", out)


def test_swiglu_quantize_equals_quantizing_the_bf16_activation(nvq):
    # the fused kernel gives the bytes of the unfused path: SwiGLU to bf16 (oracle), then the GPU's
    # own per-token quantizer
    R, I = 200, 768
    bits = _gate_up(R, I, seed=9)
    fused = nvq.nvfp4_swiglu_quantize_per_token(workloads.from_bits(bits, "cuda"))
    unfused = nvq.nvfp4_quantize_per_token(workloads.from_bits(oracle.swiglu_rows(bits), "cuda"))
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(fused, unfused))


def test_full_size_swiglu_quantize_sampled(nvq):
    # the MoE gate_up output shape: 132960 routed rows x (768 + 768)
    counts, offsets = workloads.moe_routing()
    x = workloads.routed_activations(counts, offsets, 2 * workloads.INTERMEDIATE, seed=12, device="cuda")
    q, sf, s = nvq.nvfp4_swiglu_quantize_per_token(x)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(5).choice(x.shape[0], 256, replace=False))
    xb = workloads.to_bits(x[torch.from_numpy(rows).cuda()])
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(oracle.swiglu_rows(xb))
    idx = torch.from_numpy(rows).cuda()
    assert np.array_equal(_np(q[idx]), q_ref)
    assert np.array_equal(_np(s[idx]).view(np.uint32), s_ref.view(np.uint32))
    kb = workloads.INTERMEDIATE // 16
    r_idx, c_idx = np.meshgrid(rows, np.arange(kb), indexing="ij")
    assert np.array_equal(_np(sf)[oracle.mma_layout_offset(r_idx, c_idx, kb)], sf_ref)
