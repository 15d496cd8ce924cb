"""Oracle quantisation of large operands, row chunks in parallel worker processes.

The oracle's quantisers work row by row once the NVFP4 tensor scale is known: an MXFP8 block
scale depends on its own 32 values, an NVFP4 block scale on its 16 values and the tensor scale
s.  So a matrix cut into row chunks, each chunk quantised by the oracle (NVFP4 with the s of the
whole matrix, computed by the oracle's own function), gives the oracle's bytes for the whole
matrix; ``tests/test_oracle_quantize.py`` checks that on CPU.  Workers are started with the
``spawn`` method (never forked from a process that has touched the GPU) and import only numpy
and the oracle.
"""

import multiprocessing as mp
import os

import numpy as np

from oracle import layout as L
from oracle import quantize as Q


def _quantize_chunk(args):
    kind, x, s = args
    if kind == "mxfp8":
        return Q.quantize_mxfp8(x)
    codes, sc, _ = Q.quantize_nvfp4(x, s)
    return codes, sc


def _chunks(rows, parts):
    step = max(1, -(-rows // parts))
    return [(r, min(rows, r + step)) for r in range(0, rows, step)]


def quantize_rows(kind, x, pool=None, parts=None):
    """Oracle quantisation of float32 x [rows, K] -> (codes, linear scales, s or None), the
    row chunks spread over `pool` (a multiprocessing pool) when one is given."""
    x = np.asarray(x, dtype=np.float32)
    s = Q.nvfp4_global_scale(x) if kind == "nvfp4" else None
    parts = parts or (4 * (os.cpu_count() or 1))
    jobs = [(kind, x[a:b], s) for a, b in _chunks(x.shape[0], parts)]
    res = pool.map(_quantize_chunk, jobs) if pool is not None else [_quantize_chunk(j) for j in jobs]
    codes = np.concatenate([r[0] for r in res], axis=0)
    scales = np.concatenate([r[1] for r in res], axis=0)
    return codes, scales, s


def operand(kind, x, pool=None):
    """(codes, swizzled scale buffer, s or None) of x by the oracle, as parity_util.oracle_operand."""
    codes, scales, s = quantize_rows(kind, x, pool)
    return codes, L.swizzle(scales), s


def spawn_pool(procs=None):
    """A pool of `procs` (default: the host's cores) worker processes started by spawning."""
    return mp.get_context("spawn").Pool(procs or os.cpu_count() or 1)
