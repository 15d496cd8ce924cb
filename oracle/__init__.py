"""CPU oracle of the block-scaled (MXFP8 / NVFP4) GEMM and its quantisers.

TEST INFRASTRUCTURE. A plain, slow float64 restatement of what the library
computes, written independently of the CUDA path (the two share no code).  Only
the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
use it; the product never imports it.

Pins: every function here is checked by ``tests/test_oracle_*.py`` against
facts that do not come from the oracle itself (format definitions, closed
forms, exact rational brute force, library routines on special cases).
"""

from . import formats, layout, quantize, gemm  # noqa: F401
