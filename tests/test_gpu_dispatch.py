"""GPU parity of nvfp4_quantize_dispatch (quantize-once dispatch): each routed row equals the
oracle's per-token NVFP4 of its token, byte for byte, and the whole batch equals quantizing the
tokens and gathering their rows with quantized_gather_rows. [Miles-zh = page "Miles 在 Blackwell GPU 上
实现低精度强化学习，降低训练成本", section "逐 Token 激活值缩放": one FP32 scale per token, so tokens can
be quantized once before dispatch.]"""
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
    x = rng.standard_normal((T, K)) * np.exp(rng.uniform(-4, 4, (T, 1)))
    x[rng.random((T, K)) < 0.02] *= 50.0
    x[0] = 0.0                                           # an all-zero token
    return oracle.f64_to_bf16_bits_rne(x)


def _expected(bits, dest, R, layout):
    """Oracle outputs: routed row dest[t, k] = per-token NVFP4 of token t; other rows hold the
    sentinel byte 0xAB (left as they were), MMA padding rows zero."""
    T, K = bits.shape
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(bits)
    qe = np.full((R, K // 2), 0xAB, np.uint8)
    sfe = np.full((R, K // 16), 0xAB, np.uint8)
    se = np.full(R, 0xABABABAB, np.uint32)
    t_idx, k_idx = np.nonzero(dest >= 0)
    rows = dest[t_idx, k_idx]
    qe[rows] = q_ref[t_idx]
    sfe[rows] = sf_ref[t_idx]
    se[rows] = s_ref.view(np.uint32)[t_idx]
    if layout == "mma":
        full = np.zeros(((R + 127) // 128 * 128, K // 16), np.uint8)
        full[:R] = sfe
        sfl = oracle.sf_to_mma_layout(full)
        # named rows get whole 4-column groups (zero past K/16), padding rows below R zeros, and
        # unnamed rows keep the sentinel in every byte
        off = oracle.mma_layout_offset(np.arange(R)[:, None], np.arange(((K // 16 + 3) // 4) * 4)[None, :], K // 16)
        named = np.zeros(R, bool)
        named[rows] = True
        sfl[off[~named]] = 0xAB                         # every byte of an unnamed row, padding included
        return qe, sfl, se
    return qe, sfe.reshape(-1), se


@pytest.mark.parametrize("layout", ["canonical", "mma"])
@pytest.mark.parametrize("T,K,topk,R", [(200, 272, 3, 700), (64, 2048, 8, 600), (33, 4096, 2, 70), (9, 16, 5, 50),
                                        (130, 768, 8, 1100), (8, 16384, 2, 20), (0, 64, 4, 200), (40, 96, 3, 150)])
def test_dispatch_equals_oracle(nvq, layout, T, K, topk, R):
    rng = np.random.default_rng(T + K + topk)
    bits = _tokens(T, K, T * K) if T else np.zeros((0, K), np.uint16)   # T = 0: only the padding rows
    slots = rng.permutation(R)[:T * topk]
    dest = slots.reshape(T, topk).astype(np.int32)
    dest[rng.random((T, topk)) < 0.15] = -1              # entries not dispatched
    qe, sfe, se = _expected(bits, dest, R, layout)
    lay = nvq.SF_MMA if layout == "mma" else nvq.SF_CANONICAL
    out = (torch.full((R, K // 2), 0xAB, dtype=torch.uint8, device="cuda"),
           torch.full((nvq.sf_bytes(R, K, 16, lay),), 0xAB, dtype=torch.uint8, device="cuda"),
           torch.full((R,), 0xABABABAB - 2 ** 32, dtype=torch.int32, device="cuda").view(torch.float32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, sf, s = nvq.nvfp4_quantize_dispatch(workloads.from_bits(bits, "cuda"), torch.from_numpy(dest).cuda(), R,
                                           sf_layout=layout, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == nvq.DEV_OK
    assert np.array_equal(_np(q), qe)
    assert np.array_equal(_np(s).view(np.uint32), se)
    assert np.array_equal(_np(sf).reshape(-1), sfe)


@pytest.mark.parametrize("K,pad", [(2048, 8), (272, 24)])
def test_dispatch_strided_tokens(nvq, K, pad):
    """Token rows with a pitch that is not a multiple of 16 elements (the 16-byte load path): the
    same bytes as the oracle."""
    T, topk, R = 96, 4, 500
    rng = np.random.default_rng(K + pad)
    bits = _tokens(T, K, K)
    wide = np.zeros((T, K + pad), np.uint16)
    wide[:, :K] = bits
    x = workloads.from_bits(wide, "cuda")[:, :K]
    assert x.stride(0) == K + pad and (K + pad) % 16 != 0
    dest = rng.permutation(R)[:T * topk].reshape(T, topk).astype(np.int32)
    qe, sfe, se = _expected(bits, dest, R, "mma")
    out = (torch.full((R, K // 2), 0xAB, dtype=torch.uint8, device="cuda"),
           torch.full((nvq.sf_bytes(R, K, 16),), 0xAB, dtype=torch.uint8, device="cuda"),
           torch.full((R,), 0xABABABAB - 2 ** 32, dtype=torch.int32, device="cuda").view(torch.float32))
    q, sf, s = nvq.nvfp4_quantize_dispatch(x, torch.from_numpy(dest).cuda(), R, out=out)
    torch.cuda.synchronize()
    assert np.array_equal(_np(q), qe)
    assert np.array_equal(_np(s).view(np.uint32), se)
    assert np.array_equal(_np(sf).reshape(-1), sfe)


def test_dispatch_bad_index_sets_status_and_skips_the_entry(nvq):
    T, K, R = 4, 64, 16
    bits = _tokens(T, K, 3)
    dest = np.array([[0, 1], [2, 16], [3, -7], [4, 5]], dtype=np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = (torch.zeros((R, K // 2), dtype=torch.uint8, device="cuda"),
           torch.zeros((R * K // 16,), dtype=torch.uint8, device="cuda"),
           torch.zeros((R,), dtype=torch.float32, device="cuda"))
    q, sf, s = nvq.nvfp4_quantize_dispatch(workloads.from_bits(bits, "cuda"), torch.from_numpy(dest).cuda(), R,
                                           sf_layout="canonical", out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == nvq.DEV_BAD_INDEX
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(bits)
    for t, r in [(0, 0), (0, 1), (1, 2), (2, 3), (3, 4), (3, 5)]:
        assert np.array_equal(_np(q[r]), q_ref[t])
        assert np.array_equal(_np(sf).reshape(R, -1)[r], sf_ref[t])
    assert int(q[6:].abs().sum()) == 0


@pytest.mark.parametrize("align", [1, 32])
def test_full_size_dispatch_equals_quantize_then_gather(nvq, align):
    """The MoE layer's gate_up input as the bench's default step produces it: 16384 tokens x 2048,
    top-8 of 128 experts (Zipf 1.1), routed rows unpadded (or padded to 32): the dispatch equals
    nvfp4_quantize_per_token + quantized_gather_rows on every routed row, and sampled rows equal the
    oracle."""
    T, K = 16384, workloads.HIDDEN
    choices = workloads.route_choices(T)
    counts = np.bincount(choices.reshape(-1), minlength=workloads.EXPERTS)
    offs = workloads.padded_offsets(counts, align)
    R = int(offs[-1])
    idx = torch.from_numpy(workloads.dispatch_index(choices, offs)).cuda()
    dest = torch.from_numpy(workloads.dispatch_dest(choices, offs)).cuda()
    x = workloads.normal_bf16((T, K), 1.0, seed=1, device="cuda")
    q, sf, s = nvq.nvfp4_quantize_per_token(x)
    qg, sfg, sg = nvq.quantized_gather_rows(nvq.NVFP4, q, sf, s, idx, K)
    out = (torch.zeros_like(qg), torch.zeros_like(sfg), torch.zeros_like(sg))
    qd, sfd, sd = nvq.nvfp4_quantize_dispatch(x, dest, R, out=out)
    torch.cuda.synchronize()
    assert torch.equal(qd, qg) and torch.equal(sfd, sfg) and torch.equal(sd.view(torch.int32), sg.view(torch.int32))
    rows = np.random.default_rng(5).choice(T, 48, replace=False)
    q_ref, sf_ref, s_ref = oracle.nvfp4_quantize_per_token(workloads.to_bits(x[torch.from_numpy(rows).cuda()].cpu()))
    d = _np(dest)[rows]
    for j in range(8):
        r = d[:, j]
        assert np.array_equal(_np(qd)[r], q_ref)
        assert np.array_equal(_np(sd).view(np.uint32)[r], s_ref.view(np.uint32))
        assert np.array_equal(oracle.sf_from_mma_layout(_np(sfd), R, K // 16)[r], sf_ref)
