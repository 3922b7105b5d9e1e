"""Pins for the oracle's tensor-core scale layout permutation (no GPU).

The layout itself is pinned end to end by the GPU GEMM parity tests; here: it is a bijection on
the padded tile, matches the documented in-tile offsets, and pads with zeros."""
import numpy as np

import oracle


def test_documented_offsets():
    # (row, col) -> offset within the 512-byte tile: (r%32)*16 + (r%128//32)*4 + c%4
    assert oracle.mma_layout_offset(0, 0, 4) == 0
    assert oracle.mma_layout_offset(1, 0, 4) == 16
    assert oracle.mma_layout_offset(32, 0, 4) == 4
    assert oracle.mma_layout_offset(96, 3, 4) == 15
    assert oracle.mma_layout_offset(31, 3, 4) == 31 * 16 + 3
    assert oracle.mma_layout_offset(128, 0, 4) == 512          # next row tile
    assert oracle.mma_layout_offset(0, 4, 8) == 512            # next column tile
    assert oracle.mma_layout_offset(128, 0, 8) == 1024


def test_bijection_and_round_trip():
    rng = np.random.default_rng(0)
    for rows, kb in [(128, 4), (256, 64), (300, 10), (1, 1), (129, 5)]:
        sf = rng.integers(1, 255, (rows, kb)).astype(np.uint8)
        flat = oracle.sf_to_mma_layout(sf)
        assert flat.size == oracle.mma_layout_bytes(rows, kb)
        assert flat.size == ((rows + 127) // 128 * 128) * ((kb + 3) // 4 * 4)
        assert np.array_equal(oracle.sf_from_mma_layout(flat, rows, kb), sf)
        r, c = np.meshgrid(np.arange(rows), np.arange(kb), indexing="ij")
        offs = oracle.mma_layout_offset(r, c, kb).reshape(-1)
        assert len(set(offs.tolist())) == rows * kb                 # injective
        assert (flat != 0).sum() == rows * kb                       # padding is zero
