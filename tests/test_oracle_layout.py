"""Pins of the oracle's scale-factor layout.

The pages fix the padding (rows to 128, scale columns to 4) and that the
128 x 4 blocks are interleaved; the byte map inside a block is a reading of
the public block-scaling layout that only the GPU's tensor cores can confirm
(the GEMM parity tests with per-row, per-block random scales do that).  Here:
sizes, padding, bijectivity, and that every 512-byte atom holds exactly one
128 x 4 block.
"""

import numpy as np
import pytest

from oracle import layout as L


@pytest.mark.parametrize("rows,cols", [(1, 1), (128, 4), (129, 5), (256, 8), (8000, 256), (300, 2)])
def test_padded_size(rows, cols):
    rp, cp = L.padded_shape(rows, cols)
    assert rp % 128 == 0 and cp % 4 == 0 and rp >= rows and cp >= cols
    assert rp - rows < 128 and cp - cols < 4
    assert L.sf_bytes(rows, cols) == rp * cp


@pytest.mark.parametrize("rows,cols", [(128, 4), (129, 5), (300, 10), (256, 16)])
def test_bijection_and_zero_padding(rows, cols):
    rng = np.random.default_rng(rows * 31 + cols)
    sf = rng.integers(1, 256, size=(rows, cols), dtype=np.uint8)
    buf = L.swizzle(sf)
    assert buf.size == L.sf_bytes(rows, cols)
    assert np.array_equal(L.unswizzle(buf, rows, cols), sf)
    rp, cp = L.padded_shape(rows, cols)
    r, c = np.meshgrid(np.arange(rp), np.arange(cp), indexing="ij")
    offs = L.sf_offset(r, c, cols).ravel()
    assert np.array_equal(np.sort(offs), np.arange(rp * cp))          # a permutation
    valid = ((r < rows) & (c < cols)).ravel()
    assert np.all(buf[offs[~valid]] == 0)                              # padding bytes are zero
    assert np.count_nonzero(buf) == rows * cols


def test_atoms_hold_whole_128x4_blocks():
    rows, cols = 384, 12
    rp, cp = L.padded_shape(rows, cols)
    r, c = np.meshgrid(np.arange(rp), np.arange(cp), indexing="ij")
    atom = L.sf_offset(r, c, cols) // 512
    blk = (r // 128) * (cp // 4) + (c // 4)
    assert np.array_equal(atom, blk)
    # atoms of one 128-row band are contiguous along the scale columns
    assert L.sf_offset(0, 4, cols) - L.sf_offset(0, 0, cols) == 512
    assert L.sf_offset(128, 0, cols) == (cp // 4) * 512
