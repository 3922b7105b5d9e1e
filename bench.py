"""Benchmark of the MXFP8 / per-token NVFP4 quantizer + block-scaled GEMM hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints ONE JSON line (rank 0). Workloads (synthetic, seeded; shapes of the Qwen3-30B-A3B RL workload
the pages ablate, see workloads.py):

  moe      (default) one routed MoE expert layer forward in per-token NVFP4, Qwen3-30B-A3B shapes:
           16384 tokens, top-8 of 128 experts with Zipf(1.1) loads (131072 routed rows, expert
           segments at any row): per-token NVFP4 of the routed gate_up input [R, 2048], NVFP4 of
           W_gate_up [128, 2048, 1536] and W_down [128, 768, 2048] (one FP32 scale per expert), the
           grouped gate_up GEMM, the fused SwiGLU + per-token NVFP4 of its bf16 output, and the
           grouped down GEMM.
  dense    X bf16 [8192, 2048] with per-row scales, W_qkv bf16 [2048, 5120]. One step is every
           quantizer and GEMM on that batch: MXFP8 rowwise + columnwise quantization of X, MXFP8
           columnwise quantization of W, per-token NVFP4 of X, NVFP4 of W (one matrix scope), the
           MXFP8 and the NVFP4 block-scaled GEMM (bf16 out), and the BF16 dequantization of the NVFP4
           W (dequantized-backward operand).
  backward the moe shapes in MXFP8 backward: row+col quantization of the routed X and dY, rowwise
           MXFP8 of the expert weights, grouped data-gradient GEMMs and grouped weight-gradient GEMMs.
  decode   256 tokens, uniform top-8 (2048 routed rows): per-token NVFP4 of the activations, the
           grouped NVFP4 gate_up GEMM, the fused SwiGLU + NVFP4 and the grouped NVFP4 down GEMM against
           both resident NVFP4 weight stacks, plus the BF16 dequantization of all gate_up weights.
  dq_backward  the backward shapes with the dequantized-backward mode: BF16 dequantization of the
           MXFP8 operands and grouped BF16 GEMMs.
  quant, dispatch, swiglu, weights  (GB/s lines) the quantizers alone on the routed gate_up batch;
           quantize-once dispatch (per-token NVFP4 of the tokens, each written to its routed rows);
           the fused SwiGLU + per-token NVFP4 of the down-projection input; NVFP4 quantization of all
           gate_up and down expert weights.

value = block-scaled GEMM throughput of the step (GEMM flops of the step / device time of the whole
step, quantizers included) in TFLOPS; the quantizers' GB/s and every kernel's fraction of its
roofline are in "kernels". Inputs are resident in HBM when the timed region starts; L2 is flushed
(256 MiB write) before every step, outside the step's events. "e2e" repeats the step through the
same C-ABI with host-resident (pinned) inputs copied in and the GEMM outputs copied back inside the
timed region (steps pipelined over copy-in, compute and copy-out streams). --impl reference times
the CPU oracle (test infrastructure) on a bounded sample.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantize GB/s (% HBM peak); block-scaled MoE GEMM TFLOPS (% dense peak)"
L2_FLUSH_BYTES = 256 << 20
COPY_STREAMS = 4

# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the kernels timed
# here, keyed by workload and kernel, with the sha256 of the source file (and the csrc headers) the
# capture was taken from; each figure comes from a capture of that one kernel (a launch or two,
# after the warm-up steps) of this script's own command. A changed source reports null.
NCU_TRAFFIC = {
    # the weight quantizers: amax + encode launches of one call (check, finalize and zeroing move < 0.1 MB)
    "moe": {
        "nvfp4_quantize_dispatch tokens -> routed gate_up input": {"bytes": 164628608, "src_sha": "0bcc02f7ce47fa98"},
        "nvfp4_quantize_weights gate_up": {"bytes": 1814086912, "src_sha": "43bc634262ccb6ed"},
        "block_scaled_gemm NVFP4 gate_up": {"bytes": 758438144, "src_sha": "b555bf0a103e30fb"},
        "nvfp4_swiglu_quantize_per_token down input": {"bytes": 449146368, "src_sha": "0bcc02f7ce47fa98"},
        "nvfp4_quantize_weights down": {"bytes": 888220672, "src_sha": "43bc634262ccb6ed"},
        "block_scaled_gemm NVFP4 down": {"bytes": 663508224, "src_sha": "b555bf0a103e30fb"},
    },
}


def _src_hash(name):
    """sha256 (16 hex digits) of a kernel's source file and of the csrc headers it may include."""
    csrc = os.path.join(ROOT, "nvfp4_quantization_block_gb300", "csrc")
    h = hashlib.sha256()
    for f in [name] + sorted(x for x in os.listdir(csrc) if x.endswith((".cuh", ".h"))):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------------------------------------
# CUDA path
# ------------------------------------------------------------------------------------------------
class Timer:
    """CUDA events around each named launch group on the current stream; per-step totals."""

    def __init__(self, torch):
        self.torch = torch
        self.records = {}
        self.active = False

    def run(self, name, fn):
        if not self.active:
            return fn()
        t = self.torch
        a, b = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        a.record()
        out = fn()
        b.record()
        self.records.setdefault(name, []).append((a, b))
        return out

    def durations_ms(self):
        return {k: [a.elapsed_time(b) for a, b in v] for k, v in self.records.items()}


def max_over_ranks(value_ms, world, device=None):
    """Slowest rank's time (the whole job ends when the last replica ends); plain value at world 1."""
    if world <= 1:
        return float(value_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(amount_per_step, steps, world, total_ms, scale):
    """Whole-job throughput: every rank processes its own batch (weak scaling), so the units of all
    ranks divided by the slowest rank's time; ``scale`` converts to the reported unit."""
    return amount_per_step * steps * world / (total_ms * 1e-3) / scale


class Kernel:
    """Accounting for one timed launch group: algorithmic bytes or flops per step and its roofline."""

    def __init__(self, name, bound, amount, src, peak_key, note):
        self.name, self.bound, self.amount, self.src, self.peak_key, self.note = name, bound, amount, src, peak_key, note


def _workload_dense(torch, nvq, wl, dev):
    inp = wl.dense_inputs(seed=0, device=dev)
    x, w = inp["x"], inp["w"]
    M, K = x.shape
    N = w.shape[1]
    w3 = w.unsqueeze(0).contiguous()
    offs = torch.tensor([0, M], dtype=torch.int64, device=dev)
    bufs = {
        "mx": {"q_row": torch.empty((M, K), dtype=torch.uint8, device=dev),
               "sf_row": torch.empty(nvq.sf_bytes(M, K, 32), dtype=torch.uint8, device=dev),
               "q_colT": torch.empty((K, M), dtype=torch.uint8, device=dev),
               "sf_colT": torch.empty(nvq.sf_bytes(K, M, 32), dtype=torch.uint8, device=dev)},
        "mw": {"q_colT": torch.empty((N, K), dtype=torch.uint8, device=dev),
               "sf_colT": torch.empty(nvq.sf_bytes(N, K, 32), dtype=torch.uint8, device=dev)},
        "nx": (torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
               torch.empty(nvq.sf_bytes(M, K, 16), dtype=torch.uint8, device=dev),
               torch.empty(M, dtype=torch.float32, device=dev)),
        "nw": (torch.empty((1, N, K // 2), dtype=torch.uint8, device=dev),
               torch.empty(nvq.sf_bytes(N, K, 16), dtype=torch.uint8, device=dev),
               torch.empty(1, dtype=torch.float32, device=dev)),
        "d8": torch.empty((M, N), dtype=torch.bfloat16, device=dev),
        "d4": torch.empty((M, N), dtype=torch.bfloat16, device=dev),
        "wdq": torch.empty((N, K), dtype=torch.bfloat16, device=dev),
    }
    ne_x, ne_w = M * K, K * N
    gemm_flops = 2.0 * M * N * K
    kernels = [
        Kernel("mxfp8_quantize X row+col", "hbm", ne_x * (2 + 2 * (1 + 1 / 32)), "quant_mxfp8.cu", "hbm", "4.0625 B/elem"),
        Kernel("mxfp8_quantize W col", "hbm", ne_w * (2 + 1 + 1 / 32), "quant_mxfp8.cu", "hbm", "3.03125 B/elem"),
        Kernel("nvfp4_quantize_per_token X", "hbm", ne_x * (2 + 0.5 + 1 / 16) + 4 * M, "quant_nvfp4.cu", "hbm",
               "2.5625 B/elem + 4 B/row"),
        Kernel("nvfp4_quantize_weights W", "hbm", ne_w * (2 + 0.5 + 1 / 16) + 4, "quant_nvfp4_weights.cu", "hbm",
               "2.5625 B/elem (one read; the kernel reads twice)"),
        Kernel("block_scaled_gemm MXFP8", "tensor", gemm_flops, "gemm_sm103.cu", "fp8", "2*M*N*K"),
        Kernel("block_scaled_gemm NVFP4", "tensor", gemm_flops, "gemm_sm103.cu", "fp4", "2*M*N*K"),
        Kernel("dequantize_bf16 W", "hbm", ne_w * (0.5 + 1 / 16 + 2), "dequant.cu", "hbm", "2.5625 B/elem"),
    ]

    # The timed step runs W's quantizations and the dequantization on a side stream next to X's
    # quantizations (small grids that leave the GPU partly idle on their own), joined by events
    # before the GEMMs that read them; the per-kernel pass (timer active) runs every launch in order.
    side = torch.cuda.Stream(device=dev)
    evs = [torch.cuda.Event() for _ in range(4)]

    def step(timer, xin=None, win=None):
        xx = x if xin is None else xin
        ww = w if win is None else win
        ww3 = w3 if win is None else win.unsqueeze(0)
        mx, mw, nx, nw = bufs["mx"], bufs["mw"], bufs["nx"], bufs["nw"]
        gemm8 = lambda: nvq.block_scaled_grouped_gemm(
            nvq.MXFP8, nvq.GEMM_GROUP_M, mx["q_row"], mx["sf_row"], mw["q_colT"], mw["sf_colT"], offs,
            m=M, n=N, k=K, groups=1, out=bufs["d8"])
        gemm4 = lambda: nvq.block_scaled_grouped_gemm(
            nvq.NVFP4, nvq.GEMM_GROUP_M, nx[0], nx[1], nw[0], nw[1], offs, m=M, n=N, k=K, groups=1,
            s_a=nx[2], s_b=nw[2], out=bufs["d4"])
        dq = lambda: nvq.dequantize_bf16(nvq.NVFP4, nw[0], nw[1], nw[2], nvq.SCOPE_MATRIX, groups=1, rows=N, cols=K,
                                         out=bufs["wdq"])
        if timer.active:
            timer.run(kernels[0].name, lambda: nvq.mxfp8_quantize(xx, out=bufs["mx"]))
            timer.run(kernels[1].name, lambda: nvq.mxfp8_quantize(ww, rowwise=False, out=bufs["mw"]))
            timer.run(kernels[2].name, lambda: nvq.nvfp4_quantize_per_token(xx, out=bufs["nx"]))
            timer.run(kernels[3].name, lambda: nvq.nvfp4_quantize_weights(ww3, out=bufs["nw"]))
            timer.run(kernels[4].name, gemm8)
            timer.run(kernels[5].name, gemm4)
            timer.run(kernels[6].name, dq)
            return [bufs["d8"], bufs["d4"]]
        cur = torch.cuda.current_stream(dev)
        evs[0].record(cur)
        side.wait_event(evs[0])
        with torch.cuda.stream(side):
            nvq.mxfp8_quantize(ww, rowwise=False, out=bufs["mw"])
            evs[1].record(side)
            nvq.nvfp4_quantize_weights(ww3, out=bufs["nw"])
            evs[2].record(side)
            dq()
            evs[3].record(side)
        nvq.mxfp8_quantize(xx, out=bufs["mx"])
        nvq.nvfp4_quantize_per_token(xx, out=bufs["nx"])
        cur.wait_event(evs[1])
        gemm8()
        cur.wait_event(evs[2])
        gemm4()
        cur.wait_event(evs[3])                                 # the step ends with the dequantization
        return [bufs["d8"], bufs["d4"]]

    config = {"workload": "dense linear forward, Qwen3-30B-A3B attention QKV shape (full hot path)",
              "x": [M, K], "w": [K, N], "x_rows": "N(0,1) x exp(U(ln 0.1, ln 10)) per row", "w_std": 0.02,
              "gemm_out": "bf16"}
    return {"step": step, "kernels": kernels, "gemm_flops": 2 * gemm_flops, "inputs": [x, w],
            "config": config, "dtype": "mxfp8(e4m3+e8m0)/nvfp4(e2m1+e4m3+fp32) -> fp32 accumulate -> bf16"}


def _workload_moe(torch, nvq, wl, dev, quantize_once=True, concurrent=True):
    """One routed MoE expert layer forward in per-token NVFP4: the gate_up input quantized per token,
    both expert weight matrices quantized (one FP32 scale per expert), the grouped gate_up GEMM, the
    fused SwiGLU + per-token NVFP4 of its bf16 output, and the grouped down GEMM. Expert segments
    start at any row (no padding).

    quantize_once (the default line): the layer's input is the 16384 tokens and their routing; each
    token is quantized once and written to its 8 expert-sorted routed rows by nvfp4_quantize_dispatch
    (per-token scales make this equal, byte for byte, to quantizing the gathered bf16 rows).
    Otherwise (workload moe_rows) the input is 131072 routed bf16 rows, quantized as they are."""
    import numpy as np
    T, E, H, I2, I = 16384, wl.EXPERTS, wl.HIDDEN, 2 * wl.INTERMEDIATE, wl.INTERMEDIATE
    choices = wl.route_choices(T)
    counts = np.bincount(choices.reshape(-1), minlength=E).astype(np.int64)
    offs_np = wl.padded_offsets(counts, 1)
    offs = torch.from_numpy(offs_np).to(dev)
    R = int(offs_np[-1])
    if quantize_once:
        x1 = wl.normal_bf16((T, H), 1.0, seed=1, device=dev)                 # the layer's tokens
        dest = torch.from_numpy(wl.dispatch_dest(choices, offs_np)).to(dev)  # routed row of each (token, k)
    else:
        x1 = wl.routed_activations(counts, offs_np, H, seed=1, device=dev)  # routed rows, as given
    w1 = wl.expert_weights(H, I2, seed=3, device=dev)
    w2 = wl.expert_weights(I, H, seed=4, device=dev)
    real = float(counts.sum())
    f1, f2 = 2.0 * real * I2 * H, 2.0 * real * H * I

    def alloc_tok(rows, k):
        return (torch.empty((rows, k // 2), dtype=torch.uint8, device=dev),
                torch.empty(nvq.sf_bytes(rows, k, 16), dtype=torch.uint8, device=dev),
                torch.empty(rows, dtype=torch.float32, device=dev))

    def alloc_w(e, k, n):
        return (torch.empty((e, n, k // 2), dtype=torch.uint8, device=dev),
                torch.empty(nvq.sf_bytes(e * n, k, 16), dtype=torch.uint8, device=dev),
                torch.empty(e, dtype=torch.float32, device=dev))

    b = {"a1": alloc_tok(R, H), "a2": alloc_tok(R, I), "b1": alloc_w(E, H, I2), "b2": alloc_w(E, I, H),
         "d1": torch.empty((R, I2), dtype=torch.bfloat16, device=dev),
         "d2": torch.empty((R, H), dtype=torch.bfloat16, device=dev)}
    if quantize_once:
        row_bytes = H // 2 + H // 16 + 4
        kernels = [
            Kernel("nvfp4_quantize_dispatch tokens -> routed gate_up input", "hbm", T * H * 2 + real * row_bytes,
                   "quant_nvfp4.cu", "hbm", "2 B read per token element + K/2 + K/16 + 4 B written per routed row"),
        ]
    else:
        kernels = [
            Kernel("nvfp4_quantize_per_token gate_up input", "hbm", R * H * 2.5625 + 4 * R, "quant_nvfp4.cu", "hbm",
                   "2.5625 B/elem + 4 B/row"),
        ]
    nq = len(kernels)
    kernels += [
        Kernel("nvfp4_quantize_weights gate_up", "hbm", E * H * I2 * 2.5625 + 4 * E, "quant_nvfp4_weights.cu", "hbm",
               "2.5625 B/elem"),
        Kernel("block_scaled_gemm NVFP4 gate_up", "tensor", f1, "gemm_sm103.cu", "fp4", "2*sum_e M_e*N*K"),
        Kernel("nvfp4_swiglu_quantize_per_token down input", "hbm", R * (2 * I * 2 + I / 2 + I / 16 + 4),
               "quant_nvfp4.cu", "hbm", "4 B read per h element (gate and up bf16) + 0.5625 B written + 4 B/row"),
        Kernel("nvfp4_quantize_weights down", "hbm", E * I * H * 2.5625 + 4 * E, "quant_nvfp4_weights.cu", "hbm",
               "2.5625 B/elem"),
        Kernel("block_scaled_gemm NVFP4 down", "tensor", f2, "gemm_sm103.cu", "fp4", "2*sum_e M_e*N*K"),
    ]

    # The expert-weight quantizations depend on nothing else in the step, so the timed step runs
    # them on a side stream: W_gate_up next to the activation quantization, W_down next to the
    # fused SwiGLU (after the gate_up GEMM, which holds every SM), each joined by an event before
    # the GEMM that reads it. The per-kernel pass (timer active) runs the same launches in order on
    # one stream, so each kernel's duration is its own.
    side = torch.cuda.Stream(device=dev)
    evs = [torch.cuda.Event() for _ in range(4)]

    def step(timer, xin=None, win=None):
        xa = x1 if xin is None else xin[0]
        wa, wb = (w1, w2) if win is None else win
        serial = timer.active or not concurrent
        cur = torch.cuda.current_stream(dev)

        def act():
            if quantize_once:
                timer.run(kernels[0].name, lambda: nvq.nvfp4_quantize_dispatch(xa, dest, R, out=b["a1"]))
            else:
                timer.run(kernels[0].name, lambda: nvq.nvfp4_quantize_per_token(xa, out=b["a1"]))

        def wq(k, w, out, ev_wait, ev_done):
            if serial:
                timer.run(kernels[k].name, lambda: nvq.nvfp4_quantize_weights(w, out=out))
                return
            ev_wait.record(cur)
            side.wait_event(ev_wait)
            with torch.cuda.stream(side):
                nvq.nvfp4_quantize_weights(w, out=out)
                ev_done.record(side)

        if serial:
            act()
            wq(nq, wa, b["b1"], None, None)
        else:
            wq(nq, wa, b["b1"], evs[0], evs[1])
            act()
            cur.wait_event(evs[1])
        timer.run(kernels[nq + 1].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.NVFP4, nvq.GEMM_GROUP_M, b["a1"][0], b["a1"][1], b["b1"][0], b["b1"][1], offs, m=R, n=I2, k=H,
            groups=E, s_a=b["a1"][2], s_b=b["b1"][2], out=b["d1"]))
        if serial:
            timer.run(kernels[nq + 2].name, lambda: nvq.nvfp4_swiglu_quantize_per_token(b["d1"], out=b["a2"]))
            wq(nq + 3, wb, b["b2"], None, None)
        else:
            wq(nq + 3, wb, b["b2"], evs[2], evs[3])
            nvq.nvfp4_swiglu_quantize_per_token(b["d1"], out=b["a2"])
            cur.wait_event(evs[3])
        timer.run(kernels[nq + 4].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.NVFP4, nvq.GEMM_GROUP_M, b["a2"][0], b["a2"][1], b["b2"][0], b["b2"][1], offs, m=R, n=H, k=I,
            groups=E, s_a=b["a2"][2], s_b=b["b2"][2], out=b["d2"]))
        return [b["d2"]]

    what = ("16384 tokens quantized once, each written to its 8 expert-sorted routed rows"
            if quantize_once else "the routed bf16 rows quantized as given")
    config = {"workload": "per-token NVFP4 MoE expert layer forward, Qwen3-30B-A3B shapes: 16384 tokens, "
                          "top-8 of 128 experts (Zipf 1.1 loads), 131072 routed rows; " + what +
                          ", both expert weight stacks quantized, gate_up GEMM, SwiGLU + NVFP4, down GEMM",
              "tokens": T, "hidden": H, "intermediate": I, "experts": E, "topk": 8,
              "routing": "Gumbel-top-8, p_r ~ r^-1.1", "routed_rows": int(real), "buffer_rows": R,
              "row_alignment": 1, "expert_rows_min_max": [int(counts.min()), int(counts.max())],
              "activation_input": "tokens [16384, 2048] + routing (quantize once, dispatch)" if quantize_once
              else "routed rows [131072, 2048]"}
    return {"step": step, "kernels": kernels, "gemm_flops": f1 + f2, "inputs": [x1, w1, w2],
            "input_groups": ([0], [1, 2]), "config": config,
            "dtype": "nvfp4(e2m1+e4m3+fp32) -> fp32 accumulate -> bf16"}


def _workload_moe_rows(torch, nvq, wl, dev):
    """The routed MoE layer forward with the 131072 routed bf16 rows as its input (no quantize-once
    dispatch): the per-token quantizer runs on every routed row."""
    return _workload_moe(torch, nvq, wl, dev, quantize_once=False, concurrent=False)


def _workload_backward(torch, nvq, wl, dev):
    counts, offs_np = wl.moe_routing()
    offs = torch.from_numpy(offs_np).to(dev)
    R = int(offs_np[-1])
    E, H, I2, I = wl.EXPERTS, wl.HIDDEN, 2 * wl.INTERMEDIATE, wl.INTERMEDIATE
    real = float(counts.sum())
    # layer 1 (gate_up): X1 [R, H] -> Y1 [R, I2], W1 [E, H, I2]; layer 2 (down): X2 [R, I] -> [R, H]
    x1 = wl.routed_activations(counts, offs_np, H, seed=1, device=dev)
    g1 = wl.routed_activations(counts, offs_np, I2, std=1e-3, seed=5, device=dev)
    x2 = wl.routed_activations(counts, offs_np, I, seed=2, device=dev)
    g2 = wl.routed_activations(counts, offs_np, H, std=1e-3, seed=6, device=dev)
    # dgrad needs W[e] with its rows = the layer's input features and blocks along the output dim
    w1 = wl.expert_weights(H, I2, seed=3, device=dev).view(E * H, I2)
    w2 = wl.expert_weights(I, H, seed=4, device=dev).view(E * I, H)

    def q_alloc(rows, cols, row, col):
        o = {}
        if row:
            o["q_row"] = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
            o["sf_row"] = torch.empty(nvq.sf_bytes(rows, cols, 32), dtype=torch.uint8, device=dev)
        if col:
            o["q_colT"] = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
            o["sf_colT"] = torch.empty(nvq.sf_bytes(cols, rows, 32), dtype=torch.uint8, device=dev)
        return o

    b = {"x1": q_alloc(R, H, False, True), "g1": q_alloc(R, I2, True, True), "w1": q_alloc(E * H, I2, True, False),
         "x2": q_alloc(R, I, False, True), "g2": q_alloc(R, H, True, True), "w2": q_alloc(E * I, H, True, False),
         "dx1": torch.empty((R, H), dtype=torch.bfloat16, device=dev),
         "dw1": torch.empty((E, H, I2), dtype=torch.bfloat16, device=dev),
         "dx2": torch.empty((R, I), dtype=torch.bfloat16, device=dev),
         "dw2": torch.empty((E, I, H), dtype=torch.bfloat16, device=dev)}
    f1 = 2.0 * real * H * I2
    f2 = 2.0 * real * I * H
    kernels = [
        Kernel("mxfp8_quantize X1 col", "hbm", R * H * 3.03125, "quant_mxfp8.cu", "hbm", "3.03125 B/elem"),
        Kernel("mxfp8_quantize dY1 row+col", "hbm", R * I2 * 4.0625, "quant_mxfp8.cu", "hbm", "4.0625 B/elem"),
        Kernel("mxfp8_quantize W1 row", "hbm", E * H * I2 * 3.03125, "quant_mxfp8.cu", "hbm", "3.03125 B/elem"),
        Kernel("block_scaled_gemm MXFP8 dgrad gate_up", "tensor", f1, "gemm_sm103.cu", "fp8", "2*sum_e M_e*N*K"),
        Kernel("block_scaled_gemm MXFP8 wgrad gate_up", "tensor", f1, "gemm_sm103.cu", "fp8", "2*sum_e M_e*N*K"),
        Kernel("mxfp8_quantize X2 col", "hbm", R * I * 3.03125, "quant_mxfp8.cu", "hbm", "3.03125 B/elem"),
        Kernel("mxfp8_quantize dY2 row+col", "hbm", R * H * 4.0625, "quant_mxfp8.cu", "hbm", "4.0625 B/elem"),
        Kernel("mxfp8_quantize W2 row", "hbm", E * I * H * 3.03125, "quant_mxfp8.cu", "hbm", "3.03125 B/elem"),
        Kernel("block_scaled_gemm MXFP8 dgrad down", "tensor", f2, "gemm_sm103.cu", "fp8", "2*sum_e M_e*N*K"),
        Kernel("block_scaled_gemm MXFP8 wgrad down", "tensor", f2, "gemm_sm103.cu", "fp8", "2*sum_e M_e*N*K"),
    ]

    def step(timer, xin=None, win=None):
        xa, ga, xb, gb = (x1, g1, x2, g2) if xin is None else xin
        wa, wb = (w1, w2) if win is None else win
        k = kernels
        timer.run(k[0].name, lambda: nvq.mxfp8_quantize(xa, rowwise=False, out=b["x1"]))
        timer.run(k[1].name, lambda: nvq.mxfp8_quantize(ga, out=b["g1"]))
        timer.run(k[2].name, lambda: nvq.mxfp8_quantize(wa, colwise=False, out=b["w1"]))
        timer.run(k[3].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.MXFP8, nvq.GEMM_GROUP_M, b["g1"]["q_row"], b["g1"]["sf_row"], b["w1"]["q_row"], b["w1"]["sf_row"],
            offs, m=R, n=H, k=I2, groups=E, out=b["dx1"]))
        timer.run(k[4].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.MXFP8, nvq.GEMM_GROUP_K, b["x1"]["q_colT"], b["x1"]["sf_colT"], b["g1"]["q_colT"], b["g1"]["sf_colT"],
            offs, m=H, n=I2, k=R, groups=E, out=b["dw1"]))
        timer.run(k[5].name, lambda: nvq.mxfp8_quantize(xb, rowwise=False, out=b["x2"]))
        timer.run(k[6].name, lambda: nvq.mxfp8_quantize(gb, out=b["g2"]))
        timer.run(k[7].name, lambda: nvq.mxfp8_quantize(wb, colwise=False, out=b["w2"]))
        timer.run(k[8].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.MXFP8, nvq.GEMM_GROUP_M, b["g2"]["q_row"], b["g2"]["sf_row"], b["w2"]["q_row"], b["w2"]["sf_row"],
            offs, m=R, n=I, k=H, groups=E, out=b["dx2"]))
        timer.run(k[9].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.MXFP8, nvq.GEMM_GROUP_K, b["x2"]["q_colT"], b["x2"]["sf_colT"], b["g2"]["q_colT"], b["g2"]["sf_colT"],
            offs, m=I, n=H, k=R, groups=E, out=b["dw2"]))
        return [b["dx1"], b["dw1"], b["dx2"], b["dw2"]]

    config = {"workload": "MXFP8 MoE backward (data and weight gradients of gate_up and down), Qwen3-30B-A3B",
              "tokens": 16384, "experts": E, "topk": 8, "routing": "Gumbel-top-8, p_r ~ r^-1.1",
              "routed_rows": int(real), "buffer_rows": R, "row_alignment": 32, "dy_std": 1e-3}
    return {"step": step, "kernels": kernels, "gemm_flops": 2 * (f1 + f2), "inputs": [x1, g1, x2, g2, w1, w2],
            "input_groups": ([0, 1, 2, 3], [4, 5]), "config": config,
            "dtype": "mxfp8(e4m3+e8m0) -> fp32 accumulate -> bf16"}


def _workload_dq_backward(torch, nvq, wl, dev):
    """Dequantized backward of the MoE layers: the MXFP8 copies of the backward workload (made
    untimed, as the forward would leave them) are dequantized to BF16 and the data and weight
    gradients run as BF16 grouped GEMMs on them [Miles-zh, "高精度反向和去量化反向"]."""
    counts, offs_np = wl.moe_routing()
    offs = torch.from_numpy(offs_np).to(dev)
    R = int(offs_np[-1])
    E, H, I2, I = wl.EXPERTS, wl.HIDDEN, 2 * wl.INTERMEDIATE, wl.INTERMEDIATE
    real = float(counts.sum())
    x1 = wl.routed_activations(counts, offs_np, H, seed=1, device=dev)
    g1 = wl.routed_activations(counts, offs_np, I2, std=1e-3, seed=5, device=dev)
    x2 = wl.routed_activations(counts, offs_np, I, seed=2, device=dev)
    g2 = wl.routed_activations(counts, offs_np, H, std=1e-3, seed=6, device=dev)
    w1 = wl.expert_weights(H, I2, seed=3, device=dev).view(E * H, I2)
    w2 = wl.expert_weights(I, H, seed=4, device=dev).view(E * I, H)
    q = {"x1": nvq.mxfp8_quantize(x1, rowwise=False), "g1": nvq.mxfp8_quantize(g1),
         "w1": nvq.mxfp8_quantize(w1, colwise=False), "x2": nvq.mxfp8_quantize(x2, rowwise=False),
         "g2": nvq.mxfp8_quantize(g2), "w2": nvq.mxfp8_quantize(w2, colwise=False)}
    del x1, g1, x2, g2, w1, w2

    def bf(rows, cols):
        return torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)

    # dequantized operands: dgrad A = dY rows, B = W rows; wgrad A = X^T, B = dY^T (columnwise copies)
    d = {"g1r": bf(R, I2), "w1": bf(E * H, I2), "x1t": bf(H, R), "g1t": bf(I2, R),
         "g2r": bf(R, H), "w2": bf(E * I, H), "x2t": bf(I, R), "g2t": bf(H, R),
         "dx1": bf(R, H), "dw1": torch.empty((E, H, I2), dtype=torch.bfloat16, device=dev),
         "dx2": bf(R, I), "dw2": torch.empty((E, I, H), dtype=torch.bfloat16, device=dev)}
    f1 = 2.0 * real * H * I2
    f2 = 2.0 * real * I * H
    dq = 1 + 1 / 32 + 2
    kernels = [
        Kernel("dequantize_bf16 dY1 row", "hbm", R * I2 * dq, "dequant.cu", "hbm", "3.03125 B/elem"),
        Kernel("dequantize_bf16 W1 row", "hbm", E * H * I2 * dq, "dequant.cu", "hbm", "3.03125 B/elem"),
        Kernel("grouped_gemm BF16 dgrad gate_up", "tensor", f1, "gemm_sm103.cu", "bf16", "2*sum_e M_e*N*K"),
        Kernel("dequantize_bf16 X1 col", "hbm", R * H * dq, "dequant.cu", "hbm", "3.03125 B/elem"),
        Kernel("dequantize_bf16 dY1 col", "hbm", R * I2 * dq, "dequant.cu", "hbm", "3.03125 B/elem"),
        Kernel("grouped_gemm BF16 wgrad gate_up", "tensor", f1, "gemm_sm103.cu", "bf16", "2*sum_e M_e*N*K"),
        Kernel("dequantize_bf16 dY2 row", "hbm", R * H * dq, "dequant.cu", "hbm", "3.03125 B/elem"),
        Kernel("dequantize_bf16 W2 row", "hbm", E * I * H * dq, "dequant.cu", "hbm", "3.03125 B/elem"),
        Kernel("grouped_gemm BF16 dgrad down", "tensor", f2, "gemm_sm103.cu", "bf16", "2*sum_e M_e*N*K"),
        Kernel("dequantize_bf16 X2 col", "hbm", R * I * dq, "dequant.cu", "hbm", "3.03125 B/elem"),
        Kernel("dequantize_bf16 dY2 col", "hbm", R * H * dq, "dequant.cu", "hbm", "3.03125 B/elem"),
        Kernel("grouped_gemm BF16 wgrad down", "tensor", f2, "gemm_sm103.cu", "bf16", "2*sum_e M_e*N*K"),
    ]

    def deq(src, key, rows, cols, out):
        return lambda: nvq.dequantize_bf16(nvq.MXFP8, src["q_" + key], src["sf_" + key], rows=rows, cols=cols, out=out)

    def step(timer, xin=None, win=None):
        k = kernels
        timer.run(k[0].name, deq(q["g1"], "row", R, I2, d["g1r"]))
        timer.run(k[1].name, deq(q["w1"], "row", E * H, I2, d["w1"]))
        timer.run(k[2].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.BF16, nvq.GEMM_GROUP_M, d["g1r"], None, d["w1"], None, offs, m=R, n=H, k=I2, groups=E, out=d["dx1"]))
        timer.run(k[3].name, deq(q["x1"], "colT", H, R, d["x1t"]))
        timer.run(k[4].name, deq(q["g1"], "colT", I2, R, d["g1t"]))
        timer.run(k[5].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.BF16, nvq.GEMM_GROUP_K, d["x1t"], None, d["g1t"], None, offs, m=H, n=I2, k=R, groups=E, out=d["dw1"]))
        timer.run(k[6].name, deq(q["g2"], "row", R, H, d["g2r"]))
        timer.run(k[7].name, deq(q["w2"], "row", E * I, H, d["w2"]))
        timer.run(k[8].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.BF16, nvq.GEMM_GROUP_M, d["g2r"], None, d["w2"], None, offs, m=R, n=I, k=H, groups=E, out=d["dx2"]))
        timer.run(k[9].name, deq(q["x2"], "colT", I, R, d["x2t"]))
        timer.run(k[10].name, deq(q["g2"], "colT", H, R, d["g2t"]))
        timer.run(k[11].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.BF16, nvq.GEMM_GROUP_K, d["x2t"], None, d["g2t"], None, offs, m=I, n=H, k=R, groups=E, out=d["dw2"]))
        return [d["dx1"], d["dw1"], d["dx2"], d["dw2"]]

    config = {"workload": "dequantized MoE backward: MXFP8 copies dequantized to BF16, BF16 grouped data and "
                          "weight gradients of gate_up and down, Qwen3-30B-A3B",
              "tokens": 16384, "experts": E, "topk": 8, "routed_rows": int(real), "buffer_rows": R,
              "row_alignment": 32, "dy_std": 1e-3}
    # its inputs are the forward's quantized copies already on the device: no host round trip to time
    return {"step": step, "kernels": kernels, "gemm_flops": 2 * (f1 + f2), "inputs": [], "e2e": False,
            "config": config, "dtype": "mxfp8 -> bf16 (dequantized) -> fp32 accumulate -> bf16"}


def _workload_decode(torch, nvq, wl, dev):
    """One rollout-decode pass of the MoE expert layer: 256 tokens, uniform top-8 over 128 experts
    (about 16 routed rows per expert), both NVFP4 weight stacks resident (quantized once, untimed)
    and streamed by the two grouped GEMMs, plus the dequantized-backward copy of the gate_up weights."""
    counts = wl.route_counts(256, zipf_s=0.0, seed=0)
    offs_np = wl.padded_offsets(counts, 1)                # expert segments start at any row
    offs = torch.from_numpy(offs_np).to(dev)
    R = int(offs_np[-1])
    E, H, I = wl.EXPERTS, wl.HIDDEN, wl.INTERMEDIATE
    I2 = 2 * I
    x = wl.routed_activations(counts, offs_np, H, seed=1, device=dev)
    w1 = wl.expert_weights(H, I2, seed=3, device=dev)
    wq1 = nvq.nvfp4_quantize_weights(w1)        # resident NVFP4 weights (quantized once, untimed)
    del w1
    w2 = wl.expert_weights(I, H, seed=4, device=dev)
    wq2 = nvq.nvfp4_quantize_weights(w2)
    del w2
    real = float(counts.sum())
    f1, f2 = 2.0 * real * I2 * H, 2.0 * real * H * I
    a1 = (torch.empty((R, H // 2), dtype=torch.uint8, device=dev),
          torch.empty(nvq.sf_bytes(R, H, 16), dtype=torch.uint8, device=dev),
          torch.empty(R, dtype=torch.float32, device=dev))
    d1 = torch.empty((R, I2), dtype=torch.bfloat16, device=dev)
    a2 = (torch.empty((R, I // 2), dtype=torch.uint8, device=dev),
          torch.empty(nvq.sf_bytes(R, I, 16), dtype=torch.uint8, device=dev),
          torch.empty(R, dtype=torch.float32, device=dev))
    d2 = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    wdq = torch.empty((E * I2, H), dtype=torch.bfloat16, device=dev)
    wbytes1 = E * I2 * H * (0.5 + 1 / 16) + 4 * E
    wbytes2 = E * H * I * (0.5 + 1 / 16) + 4 * E
    kernels = [
        Kernel("nvfp4_quantize_per_token decode activations", "hbm", R * H * 2.5625 + 4 * R, "quant_nvfp4.cu", "hbm", "2.5625 B/elem + 4 B/row"),
        Kernel("block_scaled_gemm NVFP4 decode gate_up", "hbm", wbytes1 + R * H * 0.5625 + real * I2 * 2, "gemm_sm103.cu", "hbm",
               "NVFP4 weight bytes + activation bytes + bf16 output (memory-bound)"),
        Kernel("nvfp4_swiglu_quantize_per_token decode down input", "hbm", R * I * 4.5625 + 4 * R, "quant_nvfp4.cu", "hbm",
               "4 B read per h element (gate and up bf16) + 0.5625 B written + 4 B/row"),
        Kernel("block_scaled_gemm NVFP4 decode down", "hbm", wbytes2 + R * I * 0.5625 + real * H * 2, "gemm_sm103.cu", "hbm",
               "NVFP4 weight bytes + activation bytes + bf16 output (memory-bound)"),
        Kernel("dequantize_bf16 gate_up weights", "hbm", E * I2 * H * (0.5625 + 2), "dequant.cu", "hbm", "2.5625 B/elem"),
    ]

    def step(timer, xin=None, win=None):
        xx = x if xin is None else xin[0]
        timer.run(kernels[0].name, lambda: nvq.nvfp4_quantize_per_token(xx, out=a1))
        timer.run(kernels[1].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.NVFP4, nvq.GEMM_GROUP_M, a1[0], a1[1], wq1[0], wq1[1], offs, m=R, n=I2, k=H, groups=E,
            s_a=a1[2], s_b=wq1[2], out=d1))
        timer.run(kernels[2].name, lambda: nvq.nvfp4_swiglu_quantize_per_token(d1, out=a2))
        timer.run(kernels[3].name, lambda: nvq.block_scaled_grouped_gemm(
            nvq.NVFP4, nvq.GEMM_GROUP_M, a2[0], a2[1], wq2[0], wq2[1], offs, m=R, n=H, k=I, groups=E,
            s_a=a2[2], s_b=wq2[2], out=d2))
        timer.run(kernels[4].name, lambda: nvq.dequantize_bf16(
            nvq.NVFP4, wq1[0], wq1[1], wq1[2], nvq.SCOPE_MATRIX, groups=E, rows=I2, cols=H, out=wdq))
        return [d2]

    config = {"workload": "rollout-decode NVFP4 MoE expert layer (256 tokens, uniform top-8): gate_up GEMM, "
                          "SwiGLU + NVFP4, down GEMM, + dequantize all gate_up weights",
              "tokens": 256, "experts": E, "routed_rows": int(real), "buffer_rows": R,
              "weights_nvfp4_mb": round((wbytes1 + wbytes2) / 1e6, 1)}
    return {"step": step, "kernels": kernels, "gemm_flops": f1 + f2, "inputs": [x], "input_groups": ([0], []),
            "config": config, "dtype": "nvfp4(e2m1+e4m3+fp32) -> fp32 accumulate -> bf16"}


def _workload_quant(torch, nvq, wl, dev):
    """Quantizers alone on a routed activation batch larger than L2 (the quantize GB/s metric)."""
    counts, offs_np = wl.moe_routing()
    R = int(offs_np[-1])
    H = wl.HIDDEN
    x = wl.routed_activations(counts, offs_np, H, seed=1, device=dev)
    mx = {"q_row": torch.empty((R, H), dtype=torch.uint8, device=dev),
          "sf_row": torch.empty(nvq.sf_bytes(R, H, 32), dtype=torch.uint8, device=dev),
          "q_colT": torch.empty((H, R), dtype=torch.uint8, device=dev),
          "sf_colT": torch.empty(nvq.sf_bytes(H, R, 32), dtype=torch.uint8, device=dev)}
    nx = (torch.empty((R, H // 2), dtype=torch.uint8, device=dev),
          torch.empty(nvq.sf_bytes(R, H, 16), dtype=torch.uint8, device=dev),
          torch.empty(R, dtype=torch.float32, device=dev))
    kernels = [
        Kernel("mxfp8_quantize X row+col", "hbm", R * H * 4.0625, "quant_mxfp8.cu", "hbm", "4.0625 B/elem"),
        Kernel("nvfp4_quantize_per_token X", "hbm", R * H * 2.5625 + 4 * R, "quant_nvfp4.cu", "hbm", "2.5625 B/elem + 4 B/row"),
    ]

    def step(timer, xin=None, win=None):
        xx = x if xin is None else xin[0]
        timer.run(kernels[0].name, lambda: nvq.mxfp8_quantize(xx, out=mx))
        timer.run(kernels[1].name, lambda: nvq.nvfp4_quantize_per_token(xx, out=nx))
        return [nx[0], nx[1], nx[2]]

    config = {"workload": "quantizers on the routed gate_up input (Qwen3-30B-A3B, 16384 tokens top-8)",
              "x": [R, H]}
    return {"step": step, "kernels": kernels, "gemm_flops": 0.0, "inputs": [x], "input_groups": ([0], []),
            "config": config, "dtype": "bf16 -> mxfp8 / nvfp4", "unit": "GB/s"}


def _workload_weights(torch, nvq, wl, dev):
    """NVFP4 expert-weight quantization alone: the MoE gate_up and down matrices of every expert."""
    E, H, I2, I = wl.EXPERTS, wl.HIDDEN, 2 * wl.INTERMEDIATE, wl.INTERMEDIATE
    w1 = wl.expert_weights(H, I2, seed=3, device=dev)
    w2 = wl.expert_weights(I, H, seed=4, device=dev)

    def alloc_w(e, k, n):
        return (torch.empty((e, n, k // 2), dtype=torch.uint8, device=dev),
                torch.empty(nvq.sf_bytes(e * n, k, 16), dtype=torch.uint8, device=dev),
                torch.empty(e, dtype=torch.float32, device=dev))

    b1, b2 = alloc_w(E, H, I2), alloc_w(E, I, H)
    kernels = [
        Kernel("nvfp4_quantize_weights gate_up", "hbm", E * H * I2 * 2.5625 + 4 * E, "quant_nvfp4_weights.cu", "hbm", "2.5625 B/elem"),
        Kernel("nvfp4_quantize_weights down", "hbm", E * I * H * 2.5625 + 4 * E, "quant_nvfp4_weights.cu", "hbm", "2.5625 B/elem"),
    ]

    def step(timer, xin=None, win=None):
        wa, wb = (w1, w2) if win is None else win
        timer.run(kernels[0].name, lambda: nvq.nvfp4_quantize_weights(wa, out=b1))
        timer.run(kernels[1].name, lambda: nvq.nvfp4_quantize_weights(wb, out=b2))
        return [b1[2], b2[2]]

    config = {"workload": "NVFP4 expert-weight quantization (Qwen3-30B-A3B MoE: gate_up and down of 128 experts)",
              "gate_up": [E, H, I2], "down": [E, I, H]}
    return {"step": step, "kernels": kernels, "gemm_flops": 0.0, "inputs": [w1, w2], "input_groups": ([], [0, 1]),
            "config": config, "dtype": "bf16 -> nvfp4 (e2m1 + e4m3 + fp32 scale per expert)", "unit": "GB/s"}


def _workload_dispatch(torch, nvq, wl, dev):
    """Quantize-once dispatch of the MoE gate_up input: per-token NVFP4 of the 16384 tokens, each
    token written to its 8 expert-sorted routed rows (nvfp4_quantize_dispatch, one pass)."""
    import numpy as np
    T, H = 16384, wl.HIDDEN
    choices = wl.route_choices(T)
    counts = np.bincount(choices.reshape(-1), minlength=wl.EXPERTS)
    offs_np = wl.padded_offsets(counts, 1)
    R = int(offs_np[-1])
    dest = torch.from_numpy(wl.dispatch_dest(choices, offs_np)).to(dev)
    x = wl.normal_bf16((T, H), 1.0, seed=21, device=dev)
    routed = (torch.empty((R, H // 2), dtype=torch.uint8, device=dev),
              torch.empty(nvq.sf_bytes(R, H, 16), dtype=torch.uint8, device=dev),
              torch.empty(R, dtype=torch.float32, device=dev))
    row_bytes = H // 2 + H // 16 + 4
    kernels = [
        Kernel("nvfp4_quantize_dispatch tokens -> routed rows", "hbm", T * H * 2 + int(counts.sum()) * row_bytes,
               "quant_nvfp4.cu", "hbm", "2 B read per token element + K/2 + K/16 + 4 B written per routed row"),
    ]

    def step(timer, xin=None, win=None):
        xx = x if xin is None else xin[0]
        timer.run(kernels[0].name, lambda: nvq.nvfp4_quantize_dispatch(xx, dest, R, out=routed))
        return [routed[0], routed[1], routed[2]]

    config = {"workload": "quantize-once dispatch: per-token NVFP4 of 16384 tokens x 2048, each token written to "
                          "its top-8 expert-sorted routed rows (Zipf 1.1)",
              "tokens": [T, H], "routed_rows": R}
    return {"step": step, "kernels": kernels, "gemm_flops": 0.0, "inputs": [x], "input_groups": ([0], []),
            "config": config, "dtype": "bf16 -> nvfp4 (dispatched)", "unit": "GB/s"}


def _workload_swiglu(torch, nvq, wl, dev):
    """The down projection's NVFP4 input straight from the gate_up GEMM output: SwiGLU + per-token
    NVFP4 in one pass over the 131072 x (768 + 768) routed activation."""
    counts, offs_np = wl.moe_routing(align=1)
    R = int(offs_np[-1])
    I = wl.INTERMEDIATE
    x = wl.routed_activations(counts, offs_np, 2 * I, seed=12, device=dev)
    out = (torch.empty((R, I // 2), dtype=torch.uint8, device=dev),
           torch.empty(nvq.sf_bytes(R, I, 16), dtype=torch.uint8, device=dev),
           torch.empty(R, dtype=torch.float32, device=dev))
    kernels = [
        Kernel("nvfp4_swiglu_quantize_per_token down input", "hbm", R * (2 * I * 2 + I / 2 + I / 16 + 4),
               "quant_nvfp4.cu", "hbm", "4 B read per h element (gate and up bf16) + 0.5625 B written + 4 B/row"),
    ]

    def step(timer, xin=None, win=None):
        xx = x if xin is None else xin[0]
        timer.run(kernels[0].name, lambda: nvq.nvfp4_swiglu_quantize_per_token(xx, out=out))
        return list(out)

    config = {"workload": "fused SwiGLU + per-token NVFP4 of the MoE gate_up output (Qwen3-30B-A3B shapes)",
              "gate_up": [R, 2 * I]}
    return {"step": step, "kernels": kernels, "gemm_flops": 0.0, "inputs": [x], "input_groups": ([0], []),
            "config": config, "dtype": "bf16 -> swiglu (fp32) -> nvfp4", "unit": "GB/s"}


WORKLOADS = {"dense": _workload_dense, "quant": _workload_quant, "moe": _workload_moe, "moe_rows": _workload_moe_rows,
             "backward": _workload_backward,
             "decode": _workload_decode, "dispatch": _workload_dispatch, "dq_backward": _workload_dq_backward,
             "swiglu": _workload_swiglu, "weights": _workload_weights}
GBS_WORKLOADS = ("quant", "dispatch", "swiglu", "weights")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"nvq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


def _peak(kind, peaks):
    if kind == "hbm":
        return peaks["hbm_gbs"], "GB/s"
    ratio = {"bf16": 1.0, "fp8": 2.0, "fp4": 6.0}[kind]   # dense FP8 = 2x BF16, FP4 = 6x BF16 on GB300
    return peaks["bf16_tflops"] * ratio, "TFLOP/s"


def run_ours(args):
    import torch
    import torch.distributed as dist

    import nvfp4_quantization_block_gb300 as nvq
    import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = _load_peaks()
    W = WORKLOADS[args.workload](torch, nvq, wl, dev)
    timer = Timer(torch)
    if args.steps is None:
        # size the timed region to ~2 s (clock sampling needs it), from one untimed probe step
        W["step"](timer)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        W["step"](timer)
        b.record()
        torch.cuda.synchronize()
        args.steps = int(max(20, min(5000, 2000.0 / max(a.elapsed_time(b), 1e-3))))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # warm-up
    for _ in range(args.warmup):
        flush.zero_()
        W["step"](timer)
    barrier()

    # timed region: K steps, one pair of CUDA events per step and nothing between the step's
    # launches (an event recorded between two kernels keeps the second from launching while the
    # first drains: 0.207 vs 0.25-0.27 ms per dense step), L2 flushed before each step
    step_ev = []
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)                              # let the sampler start before the timed region
    launches0 = nvq.launch_count()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        W["step"](timer)
        b.record()
        step_ev.append((a, b))
    barrier()
    wall = time.perf_counter() - t0
    launches = nvq.launch_count() - launches0
    # per-kernel pass: the same K steps again, with CUDA events around each launch group, for the
    # per-kernel durations and the roofline (each duration then includes its launch's latency)
    timer.active = True
    barrier()
    for _ in range(args.steps):
        flush.zero_()
        W["step"](timer)
    barrier()
    timer.active = False
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    if W.get("unit") == "GB/s":
        value = job_throughput(sum(k.amount for k in W["kernels"]), args.steps, world, total_ms, 1e9)
    else:
        value = job_throughput(W["gemm_flops"], args.steps, world, total_ms, 1e12)

    # per-kernel roofline
    durs = timer.durations_ms()
    kern = []
    for k in W["kernels"]:
        d = durs.get(k.name, [])
        avg_ms = sum(d) / len(d) if d else float("nan")
        peak, unit = _peak(k.peak_key, peaks)
        achieved = (k.amount / (avg_ms * 1e-3)) / (1e9 if unit == "GB/s" else 1e12)
        tr = NCU_TRAFFIC.get(args.workload, {}).get(k.name)
        traffic = tr["bytes"] if tr and tr.get("src_sha") == _src_hash(k.src) else None
        kern.append({"kernel": k.name, "bound": k.bound, "avg_ms": round(avg_ms, 5),
                     "share": None, "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": unit,
                     "frac": round(achieved / peak, 4), "algorithmic": k.note,
                     "amount_per_launch": k.amount, "traffic": traffic})
    kt = sum(x["avg_ms"] for x in kern)
    for x in kern:
        x["share"] = round(x["avg_ms"] / kt, 4)
    dom = max(kern, key=lambda x: x["avg_ms"])
    q = [x for x in kern if x["kernel"].startswith(("mxfp8_quantize", "nvfp4_quantize"))]
    quant_gbs = (sum(k.amount for k in W["kernels"] if any(k.name == x["kernel"] for x in q)) /
                 (sum(x["avg_ms"] for x in q) * 1e-3) / 1e9) if q else None

    # end to end: pinned host inputs copied in, step through the C-ABI, outputs copied out. Steps are
    # pipelined over three streams (inputs of step i+1 in, step i computing, outputs of step i-1 out)
    # with two workload instances and two buffer sets in rotation; every step's copies are inside
    # the timed region.
    e2e = None
    if not args.no_e2e and W.get("e2e", True):
        Ws = [W, WORKLOADS[args.workload](torch, nvq, wl, dev)]
        host_in = [t.detach().cpu().pin_memory() for t in W["inputs"]]
        dev_in = [[torch.empty_like(t) for t in W["inputs"]] for _ in range(2)]
        outs0 = W["step"](Timer(torch))
        torch.cuda.synchronize()                           # before the side streams touch the buffers
        host_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs0] for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out[0])
        groups = W.get("input_groups")
        # host<->device copies split into 64 MiB pieces over COPY_STREAMS streams each way, so that
        # several copy engines move one step's inputs and outputs at once
        s_ins = [torch.cuda.Stream() for _ in range(COPY_STREAMS)]
        s_outs = [torch.cuda.Stream() for _ in range(COPY_STREAMS)]
        s_in, s_cmp, s_out = s_ins[0], torch.cuda.Stream(), s_outs[0]
        ev_cmp, ev_out = [None, None], [[], []]

        def pieces(dst, src):
            a, b = dst.view(-1).view(torch.uint8), src.view(-1).view(torch.uint8)
            step = 64 << 20
            return [(a[o:o + step], b[o:o + step]) for o in range(0, a.numel(), step)]

        def run_step(j, din):
            if groups is None:
                return Ws[j]["step"](Timer(torch), din[0], din[1])
            xi = [din[i] for i in groups[0]]
            wi = [din[i] for i in groups[1]] or None
            return Ws[j]["step"](Timer(torch), xi, wi)

        def e2e_step(i):
            j = i & 1
            ev_ins = []
            jobs = [pc for h, dv in zip(host_in, dev_in[j]) for pc in pieces(dv, h)]
            for c, st in enumerate(s_ins):
                with torch.cuda.stream(st):
                    if ev_cmp[j] is not None:
                        st.wait_event(ev_cmp[j])           # step i-2 has finished reading set j
                    for dv, h in jobs[c::COPY_STREAMS]:
                        dv.copy_(h, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(st)
                    ev_ins.append(ev)
            with torch.cuda.stream(s_cmp):
                for ev in ev_ins:
                    s_cmp.wait_event(ev)
                for ev in ev_out[j]:
                    s_cmp.wait_event(ev)                   # step i-2's outputs have been copied out
                res = run_step(j, dev_in[j])
                ev_cmp[j] = torch.cuda.Event()
                ev_cmp[j].record(s_cmp)
            jobs = [pc for o, h in zip(res, host_out[j]) for pc in pieces(h, o)]
            ev_out[j] = []
            for c, st in enumerate(s_outs):
                with torch.cuda.stream(st):
                    st.wait_event(ev_cmp[j])
                    for h, o in jobs[c::COPY_STREAMS]:
                        h.copy_(o, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(st)
                    ev_out[j].append(ev)

        warm = max(2, args.warmup)
        for i in range(warm):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        e2e_steps = min(args.steps, 100)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_cmp)
        for st in s_ins:
            st.wait_event(a)                               # the timed copies start after a
        for i in range(warm, warm + e2e_steps):
            e2e_step(i)
        for ev in ev_out[(warm + e2e_steps - 1) & 1]:
            s_cmp.wait_event(ev)
        b.record(s_cmp)                                    # after the last step's output copies
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(a.elapsed_time(b), world, dev)
        if W.get("unit") == "GB/s":
            e2e_val = job_throughput(sum(k.amount for k in W["kernels"]), e2e_steps, world, e2e_ms, 1e9)
        else:
            e2e_val = job_throughput(W["gemm_flops"], e2e_steps, world, e2e_ms, 1e12)
        e2e = {"value": round(e2e_val, 2),
               "unit": W.get("unit", "TFLOPS"), "ms_per_step": round(e2e_ms / e2e_steps, 4), "steps": e2e_steps,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipelined": f"copy-in of step i+1 ({COPY_STREAMS} streams), compute of step i, copy-out of "
                            f"step i-1 ({COPY_STREAMS} streams)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload)

    if world > 1:
        dist.barrier()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": W.get("unit", "TFLOPS"), "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": W["dtype"], "data": "synthetic (seeded)",
            "config": dict(W["config"], parallelism=f"replicas x{world}" if world > 1 else "single GPU",
                           l2="256 MiB flush before every step, outside the step events",
                           gemm_flops_per_step=W["gemm_flops"]),
            "quantize_gbs": round(quant_gbs, 1) if quant_gbs else None,
            "quantize_frac_hbm": round(quant_gbs / peaks["hbm_gbs"], 4) if quant_gbs else None,
            "roofline": {"kernel": dom["kernel"], "bound": dom["bound"], "achieved": dom["achieved"],
                         "peak": dom["peak"], "unit": dom["unit"], "frac": dom["frac"], "traffic": dom["traffic"],
                         "peak_source": f"{peaks['source']} (bf16 burst x {'6' if 'NVFP4' in dom['kernel'] else '2'}"
                                        f" for tensor; STREAM copy for HBM)"},
            "kernels": kern,
            "kernel_timing": "per-kernel durations from a second pass of the K steps with CUDA events around "
                             "each launch group; value and ms_per_step from the K steps without them",
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": clk, "wall_s_timed_region": round(wall, 4),
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------------------
# CPU oracle (test infrastructure): cpu_baseline leg and the reference arm
# ------------------------------------------------------------------------------------------------
def _oracle_sample(workload, rows, cols):
    """Run the oracle on a bounded sample of the workload; returns (seconds, gemm flops, description)."""
    import numpy as np

    import oracle
    import workloads as wl

    rng = np.random.default_rng(0)
    t0 = time.perf_counter()
    flops = 0.0
    if workload == "dense":
        inp = wl.dense_inputs(seed=0, device="cpu")
        xb = wl.to_bits(inp["x"][:rows])
        wb = wl.to_bits(inp["w"][:, :cols].T.contiguous())          # W columns as rows
        t0 = time.perf_counter()
        mx = oracle.mxfp8_quantize(xb)
        mw = oracle.mxfp8_quantize(wb, colwise=False)
        nq, nsf, ns = oracle.nvfp4_quantize_per_token(xb)
        amax_w = np.abs(oracle.bf16_bits_to_f64(wl.to_bits(inp["w"]))).max()
        sw = oracle.nvfp4_token_scale(np.array([amax_w]))
        wq, wsf = oracle.nvfp4_quantize_rows(oracle.bf16_bits_to_f64(wb), np.repeat(sw, cols))
        a8 = oracle.deq_operand("mxfp8", mx["q_row"], mx["sf_row"])
        b8 = oracle.deq_operand("mxfp8", mw["q_row"], mw["sf_row"])
        d8, _ = oracle.grouped_gemm_reference("m", a8, b8[None], [0, rows])
        a4 = oracle.deq_operand("nvfp4", nq, nsf)
        b4 = oracle.deq_operand("nvfp4", wq, wsf)
        d4, _ = oracle.grouped_gemm_reference("m", a4, b4[None], [0, rows], ns, sw)
        oracle.dequantize_nvfp4(wq, wsf, np.repeat(sw, cols))
        K = xb.shape[1]
        flops = 2 * 2.0 * rows * cols * K
        desc = f"oracle on X rows [{rows} x {K}] and W columns [{K} x {cols}]: every quantizer, both GEMMs, dequant"
    elif workload == "dispatch":
        import torch
        K = wl.HIDDEN
        T = max(1, rows // 8)
        x = rng.standard_normal((T, K)).astype(np.float32)
        xb = wl.to_bits(torch.from_numpy(x).to(torch.bfloat16))
        idx = rng.integers(0, T, rows)
        t0 = time.perf_counter()
        q, sf, s = oracle.nvfp4_quantize_per_token(xb)
        q[idx], sf[idx], s[idx]
        flops = T * K * 2.5625 + 4 * T + 2 * rows * (K // 2 + K // 16 + 4)   # algorithmic bytes
        desc = f"oracle per-token NVFP4 of {T} tokens x {K}, gathered into {rows} rows"
    elif workload == "weights":
        import torch
        K = wl.HIDDEN
        w = (rng.standard_normal((1, K, cols)) * 0.02).astype(np.float32)
        wb = wl.to_bits(torch.from_numpy(w).to(torch.bfloat16))
        t0 = time.perf_counter()
        oracle.nvfp4_quantize_weights(wb)
        flops = K * cols * 2.5625 + 4                               # algorithmic bytes, not flops
        desc = f"oracle NVFP4 weights of one expert matrix [{K} x {cols}]"
    elif workload == "quant":
        import torch
        K = wl.HIDDEN
        x = rng.standard_normal((rows, K)).astype(np.float32)
        xb = wl.to_bits(torch.from_numpy(x).to(torch.bfloat16))
        t0 = time.perf_counter()
        oracle.mxfp8_quantize(xb)
        oracle.nvfp4_quantize_per_token(xb)
        flops = rows * K * (4.0625 + 2.5625) + 4 * rows            # algorithmic bytes, not flops
        desc = f"oracle MXFP8 row+col and per-token NVFP4 of {rows} rows x {K}"
    else:
        K = wl.HIDDEN
        N = 2 * wl.INTERMEDIATE
        cols = min(cols, N)
        x = rng.standard_normal((rows, K)).astype(np.float32)
        w = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
        import torch
        xb = wl.to_bits(torch.from_numpy(x).to(torch.bfloat16))
        wb = wl.to_bits(torch.from_numpy(w).to(torch.bfloat16))
        t0 = time.perf_counter()
        if workload == "backward":
            mx = oracle.mxfp8_quantize(xb)
            mw = oracle.mxfp8_quantize(wb[:, :cols].copy(), colwise=False)
            a = oracle.deq_operand("mxfp8", mx["q_row"], mx["sf_row"])
            b = oracle.deq_operand("mxfp8", oracle.mxfp8_quantize(np.ascontiguousarray(wb[:, :cols].T), colwise=False)["q_row"],
                                   oracle.mxfp8_quantize(np.ascontiguousarray(wb[:, :cols].T), colwise=False)["sf_row"])
            oracle.grouped_gemm_reference("m", a, b[None], [0, rows])
            del mw
        else:
            q, sf, s = oracle.nvfp4_quantize_per_token(xb)
            wq, wsf, sw = oracle.nvfp4_quantize_weights(wb[None, :, :cols].copy())
            a = oracle.deq_operand("nvfp4", q, sf)
            b = oracle.deq_operand("nvfp4", wq[0], wsf[0])
            oracle.grouped_gemm_reference("m", a, b[None], [0, rows], s, sw)
        flops = 2.0 * rows * cols * K
        desc = f"oracle on {rows} routed rows x {cols} output columns, K={K} (one expert's GEMM block + its quantizers)"
    return time.perf_counter() - t0, flops, desc


# The moe sample on all host cores: the oracle's own steps, split into independent units run by a
# pool of single-threaded worker processes. Phase 1 quantizes blocks of expert-weight columns (the
# expert's FP32 scale from its amax first), phase 2 quantizes blocks of routed rows per token and
# multiplies them by the dequantized weights. Module-level so that spawned workers can import them.
def _moe_w_unit(job):
    import numpy as np

    import oracle
    w_cols_bits, s_w = job                                 # [c, K] bf16 bits: columns of W as rows
    return oracle.nvfp4_quantize_rows(oracle.bf16_bits_to_f64(w_cols_bits), np.full(len(w_cols_bits), s_w))


def _moe_x_unit(job):
    import numpy as np

    import oracle
    xb, wq, wsf, s_w = job
    q, sf, s = oracle.nvfp4_quantize_per_token(xb)
    a = oracle.deq_operand("nvfp4", q, sf)
    b = oracle.deq_operand("nvfp4", wq, wsf)
    oracle.grouped_gemm_reference("m", a, b[None], [0, len(xb)], s, np.array([s_w], dtype=np.float32))
    return 2.0 * len(xb) * len(wq) * xb.shape[1]


def _ready(_):
    import oracle  # noqa: F401
    return os.getpid()


def _oracle_moe_parallel(rows, cols, procs):
    """Wall time of the moe oracle sample (rows routed rows x cols weight columns, K = 2048) on
    ``procs`` worker processes; returns (seconds, flops, description)."""
    import multiprocessing as mp

    import numpy as np
    import torch

    import workloads as wl
    rng = np.random.default_rng(0)
    K, N = wl.HIDDEN, 2 * wl.INTERMEDIATE
    cols = min(cols, N)
    xb = wl.to_bits(torch.from_numpy(rng.standard_normal((rows, K)).astype(np.float32)).to(torch.bfloat16))
    wb = wl.to_bits(torch.from_numpy((rng.standard_normal((K, N)) * 0.02).astype(np.float32)).to(torch.bfloat16))
    wt = np.ascontiguousarray(wb[:, :cols].T)
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs) as pool:
        pool.map(_ready, range(procs))                     # workers started and the oracle imported
        t0 = time.perf_counter()
        import oracle
        s_w = float(oracle.nvfp4_token_scale(np.abs(oracle.bf16_bits_to_f64(wt)).max()))
        parts = pool.map(_moe_w_unit, [(c, s_w) for c in np.array_split(wt, procs)])
        wq = np.concatenate([p[0] for p in parts])
        wsf = np.concatenate([p[1] for p in parts])
        flops = sum(pool.map(_moe_x_unit, [(x, wq, wsf, s_w) for x in np.array_split(xb, procs)]))
        sec = time.perf_counter() - t0
    desc = (f"oracle on {rows} routed rows x {cols} weight columns, K={K}: per-token NVFP4 of the rows, "
            f"NVFP4 of the weight columns, the GEMM block; {procs} worker processes (weight column "
            f"blocks, then row blocks)")
    return sec, flops, desc


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(workload, rows=None, cols=3072):
    """Time the oracle in child processes with BLAS threads pinned to 1: single-threaded, and (moe)
    on every host core as a pool of single-threaded workers. ``value`` / ``cores`` are the all-core
    figure where there is one, with the single-threaded one beside it."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    unit, scale = ("GB/s", 1e9) if workload in GBS_WORKLOADS else ("TFLOPS", 1e12)
    if rows is None:
        rows = 16384 if workload in ("moe", "moe_rows") else 4096     # several seconds of single-threaded oracle work

    def run(procs):
        cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", workload, "--rows", str(rows),
               "--cols", str(cols), "--procs", str(procs)]
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900)
        res = json.loads(out.stdout.strip().splitlines()[-1])
        return {"value": res["flops"] / res["seconds"] / scale, "unit": unit, "cores": procs, "kind": "oracle",
                "sample": res["sample"], "seconds": round(res["seconds"], 3)}

    try:
        single = run(1)
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"value": None, "unit": unit, "cores": 1, "kind": "oracle", "sample": f"failed: {e}"}
    cores = _host_cores()
    if workload not in ("moe", "moe_rows") or cores <= 1:
        return single
    try:
        allc = run(cores)
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        return dict(single, all_cores=f"failed: {e}")
    return dict(allc, single_thread={k: single[k] for k in ("value", "cores", "seconds", "sample")})


def run_reference(args):
    # the oracle runs single-threaded (numpy is first imported below, after this)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    if args.steps is None:
        args.steps = 5
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    rows, cols = 256, 256
    for _ in range(args.warmup):
        _oracle_sample(args.workload, rows, cols)
    times, flops, desc = [], 0.0, ""
    for _ in range(args.steps):
        t, flops, desc = _oracle_sample(args.workload, rows, cols)
        times.append(t)
    total = sum(times)
    unit = "GB/s" if args.workload in GBS_WORKLOADS else "TFLOPS"
    value = flops * len(times) / total / (1e9 if unit == "GB/s" else 1e12)
    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * total / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
            "impl": "reference",
            "config": {"workload": args.workload, "sample": desc},
            "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for about 2 s of device time, at least 20)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="moe")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--rows", type=int, default=512, help=argparse.SUPPRESS)
    ap.add_argument("--cols", type=int, default=512, help=argparse.SUPPRESS)
    ap.add_argument("--procs", type=int, default=1, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample:
        if args.procs > 1 and args.oracle_sample == "moe":
            t, f, d = _oracle_moe_parallel(args.rows, args.cols, args.procs)
        else:
            t, f, d = _oracle_sample(args.oracle_sample, args.rows, args.cols)
        print(json.dumps({"seconds": t, "flops": f, "sample": d}))
        return
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
