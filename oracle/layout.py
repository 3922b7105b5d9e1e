"""Tensor-core tile layout of block scales ("the layout the MMA consumes").

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The method statement asks for scale stores "in the layout the MMA consumes", and the pages warn
that backend-specific swizzled layouts must stay explicit and verifiable [Miles-zh, "重构权重更新
接口"; Miles-fr, "Ce que l'ablation Qwen3 ne démontre pas", paragraph on weight movement]. The
pages do not define the layout; it comes from the tcgen05 block-scaling description of the PTX ISA:
a scale matrix [rows, kb] (one byte per block) is cut into tiles of 128 rows x 4 scale columns;
each tile is 512 contiguous bytes in which the scale of (row r, column c) sits at
    (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4,
i.e. 32 lines of 16 bytes, line i holding rows i, i+32, i+64, i+96. Tiles are stored row-tile
major: tile (rt, ct) starts at (rt * ceil(kb/4) + ct) * 512. Rows are padded to a multiple of 128
and scale columns to a multiple of 4; padding bytes are zero.

Pinning: this permutation is checked here only for being a bijection with the documented tile
offsets (tests/test_oracle_layout.py). Its agreement with what the tensor cores consume is pinned
end to end by the GPU GEMM parity tests, where the oracle GEMM uses canonical scales only.
"""

import numpy as np


def _pad(n, m):
    return (n + m - 1) // m * m


def mma_layout_bytes(rows, kb):
    """Bytes of the tile layout for a [rows, kb] scale matrix."""
    return _pad(rows, 128) * _pad(kb, 4)


def mma_layout_offset(r, c, kb):
    """Byte offset of scale (r, c) in the tile layout of a [rows, kb] scale matrix."""
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    tiles_per_row = _pad(kb, 4) // 4
    tile = (r // 128) * tiles_per_row + c // 4
    return tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def sf_to_mma_layout(sf):
    """Canonical scales [rows, kb] (uint8) -> flat tile layout (uint8, zero padding)."""
    sf = np.asarray(sf, dtype=np.uint8)
    rows, kb = sf.shape
    out = np.zeros(mma_layout_bytes(rows, kb), dtype=np.uint8)
    r, c = np.meshgrid(np.arange(rows), np.arange(kb), indexing="ij")
    out[mma_layout_offset(r, c, kb)] = sf
    return out


def sf_from_mma_layout(flat, rows, kb):
    """Inverse of ``sf_to_mma_layout``."""
    flat = np.asarray(flat, dtype=np.uint8).reshape(-1)
    r, c = np.meshgrid(np.arange(rows), np.arange(kb), indexing="ij")
    return flat[mma_layout_offset(r, c, kb)]
