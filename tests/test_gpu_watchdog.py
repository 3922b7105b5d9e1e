"""The GEMM's bounded pipeline waits, exercised on the GPU without faulting or hanging it.

Every wait between the kernel's roles (TMA producer, scale copier, MMA issuer, epilogue) gives up
after ``wait_limit_ns``: it sets the status word to NVQ_DEV_TIMEOUT, the other roles leave their
loops, every role drains the asynchronous work it issued, and the CTA frees its tensor memory and
returns. The test makes one wait run out with the library's injection hook (the first CTA's
producer never arms one load stage, so the waits on that stage cannot complete), checks the
status, then runs a normal GEMM on the same stream and checks it against the oracle: had the
aborted CTA kept its tensor memory, the next launch could not allocate it.
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


def _operands(nvq, fmt, M, K, N, seed):
    rng = np.random.default_rng(seed)
    xb = oracle.f64_to_bf16_bits_rne(rng.standard_normal((M, K)))
    wb = oracle.f64_to_bf16_bits_rne(rng.standard_normal((1, K, N)) * 0.02)
    x, w = workloads.from_bits(xb, "cuda"), workloads.from_bits(wb, "cuda")
    if fmt == "nvfp4":
        qa, sfa, sa = nvq.nvfp4_quantize_per_token(x)
        qb, sfb, sb = nvq.nvfp4_quantize_weights(w.contiguous())
        call = (nvq.NVFP4, nvq.GEMM_GROUP_M, qa, sfa, qb, sfb), dict(s_a=sa, s_b=sb)
        qa_r, sfa_r, sa_r = oracle.nvfp4_quantize_per_token(xb)
        qb_r, sfb_r, sb_r = oracle.nvfp4_quantize_weights(wb)
        D, bound = oracle.grouped_gemm_reference("m", oracle.deq_operand("nvfp4", qa_r, sfa_r),
                                                 oracle.deq_operand("nvfp4", qb_r[0], sfb_r[0])[None],
                                                 [0, M], sa_r, sb_r)
    elif fmt == "mxfp8":
        qa = nvq.mxfp8_quantize(x, colwise=False)
        qb = nvq.mxfp8_quantize(w[0], rowwise=False)           # columnwise of W: [N, K]
        call = (nvq.MXFP8, nvq.GEMM_GROUP_M, qa["q_row"], qa["sf_row"], qb["q_colT"], qb["sf_colT"]), {}
        ra = oracle.mxfp8_quantize(xb, colwise=False)
        rb = oracle.mxfp8_quantize(np.ascontiguousarray(wb[0]), rowwise=False)
        D, bound = oracle.grouped_gemm_reference("m", oracle.deq_operand("mxfp8", ra["q_row"], ra["sf_row"]),
                                                 oracle.deq_operand("mxfp8", rb["q_colT"], rb["sf_colT"])[None],
                                                 [0, M])
    else:
        wt = w[0].T.contiguous()                               # B [N, K]
        call = (nvq.BF16, nvq.GEMM_GROUP_M, x, None, wt, None), {}
        D, bound = oracle.grouped_gemm_reference("m", oracle.bf16_bits_to_f64(xb),
                                                 oracle.bf16_bits_to_f64(np.ascontiguousarray(wb[0].T))[None],
                                                 [0, M])
    return call, D, bound


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8", "bf16"])
@pytest.mark.parametrize("stage", [1, 3])
def test_wait_that_runs_out_sets_status_and_frees_the_gpu(nvq, fmt, stage):
    M, K, N = 1024, 1024, 512                   # 16 tiles of 128 x 256, several load stages each
    (args, kw), D, bound = _operands(nvq, fmt, M, K, N, seed=stage)
    offs = torch.tensor([0, M], dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nvq.block_scaled_grouped_gemm(*args, offs, m=M, n=N, k=K, groups=1, out_type=nvq.OUT_F32, status=status,
                                  wait_limit_ns=2_000_000, inject_timeout_stage=stage, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == nvq.DEV_TIMEOUT
    # the same GEMM again on the same stream, without the injection: complete and within tolerance
    status.zero_()
    d = nvq.block_scaled_grouped_gemm(*args, offs, m=M, n=N, k=K, groups=1, out_type=nvq.OUT_F32, status=status,
                                      **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == nvq.DEV_OK
    err = np.abs(d.cpu().numpy().astype(np.float64) - D)
    assert (err <= 2e-3 * bound).all()


@pytest.mark.parametrize("stage", [1, 4])
def test_wait_that_runs_out_in_the_few_rows_per_group_layout(nvq, stage):
    # 8 experts of 24 rows each: every tile starts inside a scale tile (the transposer's waits too)
    E, rows, K, N = 8, 24, 1024, 256
    rng = np.random.default_rng(40 + stage)
    xb = oracle.f64_to_bf16_bits_rne(rng.standard_normal((E * rows, K)))
    wb = oracle.f64_to_bf16_bits_rne(rng.standard_normal((E, K, N)) * 0.02)
    qa, sfa, sa = nvq.nvfp4_quantize_per_token(workloads.from_bits(xb, "cuda"))
    qb, sfb, sb = nvq.nvfp4_quantize_weights(workloads.from_bits(wb, "cuda").contiguous())
    offs_np = np.arange(E + 1, dtype=np.int64) * rows
    offs = torch.from_numpy(offs_np).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    call = (nvq.NVFP4, nvq.GEMM_GROUP_M, qa, sfa, qb, sfb, offs)
    nvq.block_scaled_grouped_gemm(*call, m=E * rows, n=N, k=K, groups=E, s_a=sa, s_b=sb, out_type=nvq.OUT_F32,
                                  status=status, wait_limit_ns=2_000_000, inject_timeout_stage=stage)
    torch.cuda.synchronize()
    assert int(status.item()) == nvq.DEV_TIMEOUT
    status.zero_()
    d = nvq.block_scaled_grouped_gemm(*call, m=E * rows, n=N, k=K, groups=E, s_a=sa, s_b=sb, out_type=nvq.OUT_F32,
                                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == nvq.DEV_OK
    q_r, sf_r, s_r = oracle.nvfp4_quantize_per_token(xb)
    wq_r, wsf_r, ws_r = oracle.nvfp4_quantize_weights(wb)
    b = np.stack([oracle.deq_operand("nvfp4", wq_r[e], wsf_r[e]) for e in range(E)])
    D, bound = oracle.grouped_gemm_reference("m", oracle.deq_operand("nvfp4", q_r, sf_r), b, offs_np, s_r, ws_r)
    assert (np.abs(d.cpu().numpy().astype(np.float64) - D) <= 2e-3 * bound).all()
