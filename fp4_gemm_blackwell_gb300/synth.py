"""Seeded synthetic inputs for the block-scaled GEMM.

This module only draws random numbers; it holds none of the method's
arithmetic (no quantising, no scaling rule, no GEMM), so both the CUDA path's
tests and the CPU oracle can take their inputs from it.

Recipe (the workloads of the block-scaled GEMM pages, drawn with a CPU
``torch.Generator``):
* ``normal``: float32 N(0, 1), row-major (rows x cols);
* ``normal_rowscaled``: N(0, 1) times one U(0.5, 2) multiplier per row, drawn
  after the matrix from the same generator;
* ``bias``: N(0, 1) * std, rounded to the output type (bf16 or f16), returned as
  its 16-bit patterns and as float64 values;
* ``as_bf16_bits``: a float32 matrix rounded to BF16 (torch's round to nearest even),
  returned as 16-bit patterns: the input of the BF16 quantiser.
Seeds: A = 0, B = 1, bias = 2 unless a caller says otherwise.
"""

import numpy as np
import torch

SEED_A = 0
SEED_B = 1
SEED_BIAS = 2


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(rows, cols, seed):
    g = _gen(seed)
    return torch.randn((rows, cols), generator=g, dtype=torch.float32).numpy()


def normal_rowscaled(rows, cols, seed):
    g = _gen(seed)
    x = torch.randn((rows, cols), generator=g, dtype=torch.float32)
    u = torch.rand((rows, 1), generator=g, dtype=torch.float32) * 1.5 + 0.5
    return (x * u).numpy()


def bias(n, seed=SEED_BIAS, std=0.1, out="bf16"):
    g = _gen(seed)
    b = torch.randn((n,), generator=g, dtype=torch.float32) * std
    t = b.to(torch.bfloat16 if out == "bf16" else torch.float16)
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    return bits, t.to(torch.float64).numpy()


def as_bf16_bits(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()
