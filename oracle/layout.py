"""Scale-factor matrix layout: linear (rows x blocks) <-> padded, swizzled 128x4 atoms.

TEST INFRASTRUCTURE (part of the CPU oracle; see ``oracle/formats.py``).

"Add Cutlass MxFp8 Block Scale Matrix Multiplication" says the block scales are
"stored in an interleaved/swizzled layout", padded to 128 x 4 blocks (its
validation step "scales must be padded/swizzled to 128x4 blocks", its test
helper ``linear_to_swizzled_128_4`` and the comment "Scale Factor tensors have an
interleaved layout").  The page gives no byte map.  The reading taken here is the
public cuBLAS / PTX block-scaling layout:

* the rows are padded to Rp = 128 * ceil(rows / 128) and the scale columns to
  Cp = 4 * ceil(cols / 4), padding bytes 0;
* the matrix is cut into 128-row x 4-column atoms of 512 bytes, stored atom row
  by atom row ((r // 128) major, (c // 4) minor);
* inside an atom, scale (r, c) sits at byte (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4).
"""

import numpy as np


def padded_shape(rows, cols):
    """(Rp, Cp): rows padded to a multiple of 128, scale columns to a multiple of 4."""
    return ((rows + 127) // 128) * 128, ((cols + 3) // 4) * 4


def sf_bytes(rows, cols):
    rp, cp = padded_shape(rows, cols)
    return rp * cp


def sf_offset(r, c, cols):
    """Byte offset of scale (r, c) in the swizzled buffer of a matrix with ``cols`` scale columns."""
    _, cp = padded_shape(1, cols)
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    atom = (r // 128) * (cp // 4) + (c // 4)
    return atom * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def swizzle(sf_linear):
    """uint8 [rows, cols] -> uint8 [Rp * Cp] swizzled buffer (padding zero)."""
    sf_linear = np.asarray(sf_linear, dtype=np.uint8)
    rows, cols = sf_linear.shape
    out = np.zeros(sf_bytes(rows, cols), dtype=np.uint8)
    r, c = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    out[sf_offset(r, c, cols)] = sf_linear
    return out


def unswizzle(buf, rows, cols):
    """Inverse of :func:`swizzle` on the valid region."""
    buf = np.asarray(buf, dtype=np.uint8)
    if buf.size < sf_bytes(rows, cols):
        raise ValueError("scale buffer smaller than the padded 128x4 layout")
    r, c = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    return buf[sf_offset(r, c, cols)]
