"""Seeded synthetic inputs shaped like the pages' Qwen3-30B-A3B MoE workload.

This module only draws random numbers and lays them out; it holds none of the quantizer or GEMM
arithmetic, so both the CUDA path's tests/benchmark and the CPU oracle may use it.

[Miles-zh] is the page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本" (a Chinese translation of
the Miles post on Blackwell-native MXFP8 / NVFP4 RL). The pages' workload is Qwen3-30B-A3B RL on dapo-math-17k [Miles-zh, "结果：在 8x B200 上对 Qwen3-30B-A3B
配方进行消融实验"]; no dataset or checkpoint is used here. Inputs stand in for it with the model's
shapes: hidden 2048, 128 routed experts, top-8 routing, expert intermediate 768 (gate and up
concatenated: 1536), attention QKV projection 2048 -> 5120. Recipes (all bf16 = round-to-nearest of
an fp32 draw):

  contract:   X [256, 512] ~ N(0, 1) with exactly 1% of entries (drawn without replacement) x100;
              W [512, 384] ~ N(0, 0.02).
  dense:      X [8192, 2048] ~ N(0, 1) times a per-row factor exp(U(ln 0.1, ln 10));
              W_qkv [2048, 5120] ~ N(0, 0.02).
  moe:        16384 tokens; each picks 8 distinct experts of 128 by Gumbel-top-8 on log p_r with
              p_r ~ r^-1.1 (a Zipf(1.1) load profile); routed rows are contiguous per expert, each
              expert's segment padded with zero rows to a multiple of ``align`` rows.
              X_routed [rows, 2048] ~ N(0, 1); down-projection input [rows, 768] ~ N(0, 1);
              W_gate_up [128, 2048, 1536] and W_down [128, 768, 2048] ~ N(0, 0.02);
              upstream gradients dY ~ N(0, 1e-3).
  decode:     256 tokens, top-8 of 128 experts with uniform probabilities (about 16 rows each).
"""

import numpy as np
import torch

HIDDEN = 2048
EXPERTS = 128
TOPK = 8
INTERMEDIATE = 768
QKV_OUT = 5120


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std=1.0, seed=0, device="cpu"):
    """bf16 tensor ~ N(0, std) (fp32 draw rounded to bf16)."""
    g = _gen(device, seed)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def to_bits(t):
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(bits, device="cpu"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


# ----------------------------------------------------------------------------------------------
# Routing
# ----------------------------------------------------------------------------------------------

def route_choices(tokens, experts=EXPERTS, topk=TOPK, zipf_s=1.1, seed=0):
    """The ``topk`` distinct experts of every token, by Gumbel-top-k on log p_r: int64 [tokens, topk].

    zipf_s > 0: p_r ~ r^-s (r = 1..experts); zipf_s == 0: uniform.
    """
    rng = np.random.default_rng(seed)
    logp = -zipf_s * np.log(np.arange(1, experts + 1, dtype=np.float64))
    out = np.empty((tokens, topk), dtype=np.int64)
    chunk = 4096
    for t0 in range(0, tokens, chunk):
        n = min(chunk, tokens - t0)
        gumbel = -np.log(-np.log(rng.random((n, experts))))
        out[t0:t0 + n] = np.argpartition(-(logp + gumbel), topk - 1, axis=1)[:, :topk]
    return out


def route_counts(tokens, experts=EXPERTS, topk=TOPK, zipf_s=1.1, seed=0):
    """Rows per expert of ``route_choices``: int64 [experts]."""
    top = route_choices(tokens, experts, topk, zipf_s, seed)
    return np.bincount(top.reshape(-1), minlength=experts).astype(np.int64)


def dispatch_index(choices, offsets, experts=EXPERTS):
    """Source token of every routed row (expert-sorted, each expert's tokens in token order, segments
    starting at ``offsets``): int32 [offsets[-1]], -1 on padding rows."""
    choices = np.asarray(choices)
    tokens, topk = choices.shape
    idx = np.full(int(offsets[-1]), -1, dtype=np.int32)
    flat_e = choices.reshape(-1)
    flat_t = np.repeat(np.arange(tokens, dtype=np.int32), topk)
    order = np.argsort(flat_e, kind="stable")           # by expert, tokens in order within one
    counts = np.bincount(flat_e, minlength=experts)
    pos = 0
    for e in range(experts):
        c = int(counts[e])
        idx[int(offsets[e]):int(offsets[e]) + c] = flat_t[order[pos:pos + c]]
        pos += c
    return idx


def dispatch_dest(choices, offsets, experts=EXPERTS):
    """Routed row of every (token, k) of ``choices`` in the layout of ``dispatch_index`` (expert-sorted,
    each expert's tokens in token order, segments starting at ``offsets``): int32 [tokens, topk]."""
    choices = np.asarray(choices)
    tokens, topk = choices.shape
    flat_e = choices.reshape(-1)
    order = np.argsort(flat_e, kind="stable")
    counts = np.bincount(flat_e, minlength=experts)
    dest = np.empty(flat_e.size, dtype=np.int32)
    pos = 0
    for e in range(experts):
        c = int(counts[e])
        dest[order[pos:pos + c]] = np.arange(int(offsets[e]), int(offsets[e]) + c, dtype=np.int32)
        pos += c
    return dest.reshape(tokens, topk)


def padded_offsets(counts, align):
    """Segment starts [E+1]: each expert's rows padded up to a multiple of ``align``."""
    c = np.asarray(counts, dtype=np.int64)
    padded = (c + align - 1) // align * align
    return np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)


def valid_row_mask(counts, offsets):
    """Boolean [offsets[-1]]: True on real routed rows, False on padding rows."""
    m = np.zeros(int(offsets[-1]), dtype=bool)
    for e, c in enumerate(counts):
        m[offsets[e]:offsets[e] + c] = True
    return m


def zero_padding_rows(t, counts, offsets):
    """Zero the padding rows of a routed [rows, ...] tensor in place."""
    for e, c in enumerate(counts):
        s0, s1 = int(offsets[e] + c), int(offsets[e + 1])
        if s1 > s0:
            t[s0:s1] = 0
    return t


# ----------------------------------------------------------------------------------------------
# Configurations
# ----------------------------------------------------------------------------------------------

def contract_inputs(seed=0, device="cpu", rows=256, cols=512, n=384):
    x = normal_bf16((rows, cols), 1.0, seed, device).float()
    rng = np.random.default_rng(seed + 1)
    idx = rng.choice(rows * cols, size=int(round(0.01 * rows * cols)), replace=False)
    flat = x.view(-1)
    flat[torch.from_numpy(idx).to(device)] *= 100.0
    w = normal_bf16((cols, n), 0.02, seed + 2, device)
    return {"x": x.to(torch.bfloat16), "w": w}


def dense_inputs(seed=0, device="cpu", m=8192, k=HIDDEN, n=QKV_OUT):
    x = normal_bf16((m, k), 1.0, seed, device).float()
    g = _gen(device, seed + 3)
    u = torch.rand(m, 1, generator=g, device=device, dtype=torch.float64)
    lo, hi = np.log(0.1), np.log(10.0)
    x = (x.double() * torch.exp(lo + (hi - lo) * u)).to(torch.bfloat16)
    w = normal_bf16((k, n), 0.02, seed + 4, device)
    return {"x": x, "w": w}


def moe_routing(tokens=16384, zipf_s=1.1, align=32, seed=0):
    counts = route_counts(tokens, zipf_s=zipf_s, seed=seed)
    offsets = padded_offsets(counts, align)
    return counts, offsets


def routed_activations(counts, offsets, k, std=1.0, seed=0, device="cpu"):
    t = normal_bf16((int(offsets[-1]), k), std, seed, device)
    return zero_padding_rows(t, counts, offsets)


def expert_weights(k, n, experts=EXPERTS, seed=0, device="cpu"):
    """[experts, k, n] bf16 ~ N(0, 0.02) (Y = X W per expert)."""
    return normal_bf16((experts, k, n), 0.02, seed, device)
