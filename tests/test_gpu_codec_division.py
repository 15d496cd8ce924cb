"""The NVFP4 block encoder's division-free quotients against CUDA's IEEE division.

The encoder (the quantiser and the GEMM's NVFP4-output epilogue) rounds each block's amax / d and
each element's x / den to float32 before converting them to UE4M3 and E2M1 codes.  It forms those
quotients without a division, by Markstein's correction step on the correctly rounded reciprocal,
for divisors in [2^-64, 2^64] and quotients below about 2^64.  The probe
(``csrc/division_probe.cu``) draws 2^29 dividends per seed, two per divisor, a quarter of them
within a few ulps of a value where a code changes, and counts where the encoder's quotient differs
from ``__fdiv_rn``: in the float32 bits for every quotient at or above 2^-39, and in the E2M1 and
E4M3 codes for all of them.  The bit-exact quantiser tests check the whole encoder against the
oracle on realistic data; this test covers the rounding step on inputs those tensors rarely reach.
"""

import ctypes
import os

import pytest
import torch

pytestmark = pytest.mark.gpu

PROBE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc", "libdivision_probe.so")


@pytest.mark.parametrize("seed", [1, 2])
def test_markstein_quotients_match_ieee_division(seed):
    lib = ctypes.CDLL(PROBE)
    lib.division_probe.restype = ctypes.c_int
    lib.division_probe.argtypes = [ctypes.c_ulonglong, ctypes.c_ulonglong, ctypes.c_void_p, ctypes.c_void_p]
    out = torch.zeros(5, dtype=torch.int64, device="cuda")
    n = 1 << 29
    assert lib.division_probe(n, seed, out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    tested, qbad, cbad, xb, yb = (int(v) for v in out.cpu())
    assert tested > n // 2, "too few pairs inside the encoder's range: %d of %d" % (tested, n)
    assert qbad == 0 and cbad == 0, "%d quotient and %d code mismatches, e.g. x bits %#x y bits %#x" % (
        qbad, cbad, xb, yb)
