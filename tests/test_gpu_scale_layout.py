"""The scale atoms' byte order (the 128x4 layout) against the hardware and against cuBLAS.

The pages name the layout only ("interleaved/swizzled", "padded to 128x4 blocks",
``linear_to_swizzled_128_4`` in the test of "Add Cutlass MxFp8 Block Scale Matrix
Multiplication"); the oracle, the quantisers and the kernels' scale warps all follow one reading
of it: scale (r, c) at byte (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4 of its 512-byte atom.
Two checks tie that reading to something outside this library:

1. the hardware: ``tcgen05.cp`` with the 32x128b.warpx4 shape, the tensor cores' own way to load
   a scale atom, places shared-memory row i (16 bytes) of an atom into lane i of every 32-lane
   quarter of tensor memory as four 32-bit columns.  The probe copies an atom of random bytes
   and reads the lanes back; the scale warps of the GEMM kernels write that placement (lane i,
   column k = word k of atom row i; for B in every quarter, for A only the column the MMA reads
   in each quarter, k = q), so with the GEMM parity tests, whose per-block scales vary, the
   oracle's byte order is the one the tensor cores consume;
2. cuBLAS through ``torch._scaled_mm`` (where the installed PyTorch supports block-scaled
   operands on this GPU): the same codes and scale bytes, given to a second implementation of
   the published layout, must give the oracle's result; with the atom's row groups read in the
   other order the oracle's result must be far off, so the check can tell the two apart.
"""

import ctypes
import os

import numpy as np
import pytest
import torch

import parity_util as P
from oracle import gemm as R
from oracle import layout as L
from oracle import quantize as Q

pytestmark = pytest.mark.gpu

PROBE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc", "libsf_atom_probe.so")


def test_tcgen05_cp_places_atom_rows_as_the_scale_warps_do():
    lib = ctypes.CDLL(PROBE)
    lib.sf_atom_probe.restype = ctypes.c_int
    lib.sf_atom_probe.argtypes = [ctypes.c_void_p] * 4
    rng = np.random.default_rng(5)
    for _ in range(3):
        atom = rng.integers(0, 256, 512, dtype=np.uint8)
        a = torch.from_numpy(atom).cuda()
        out = torch.zeros(128 * 4, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        assert lib.sf_atom_probe(a.data_ptr(), out.data_ptr(), status.data_ptr(), stream) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0, "the copy's completion was not seen"
        got = out.cpu().numpy().view(np.uint32).reshape(4, 32, 4)       # [quarter][lane][column]
        words = atom.view("<u4").reshape(32, 4)                          # [atom row][word]
        for q in range(4):
            assert np.array_equal(got[q], words), "lane quarter %d" % q


def _blocky(rows, K, blk, seed, lo, hi):
    """N(0, 1) values times 2^e per (row, block), e uniform in [lo, hi]: block scales that differ
    from block to block, so that any other placement of the scale bytes changes the result."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, K)).astype(np.float32)
    e = rng.integers(lo, hi + 1, (rows, K // blk))
    return (x * np.repeat(np.ldexp(1.0, e), blk, axis=1)).astype(np.float32)


def _other_order(sf_lin, rows, cols):
    """The same scales with each 512-byte atom laid out as plain row-major 128 x 4 bytes (scale
    (r, c) at byte (r % 128) * 4 + c % 4 of its atom): the plainest other reading of "128x4"."""
    buf = L.swizzle(sf_lin).reshape(-1, 512).copy()
    out = np.empty_like(buf)
    rr = np.arange(128)
    src = (rr % 32) * 16 + (rr // 32) * 4
    dst = rr * 4
    for c in range(4):
        out[:, dst + c] = buf[:, src + c]
    return out.reshape(-1)


def _scaled_mm(a_t, b_t, sa, sb):
    try:
        return torch._scaled_mm(a_t, b_t.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)
    except (RuntimeError, TypeError, NotImplementedError) as e:
        pytest.skip("torch._scaled_mm has no block-scaled path for this here: %s" % str(e).splitlines()[0][:160])


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_scale_layout_matches_cublas(kind):
    M, N, K = 256, 384, 512
    blk = 32 if kind == "mxfp8" else 16
    # UE8M0 scales span the exponents at will; UE4M3 ones (tensor scale 1) stay within range
    lo, hi = (-10, 10) if kind == "mxfp8" else (-6, 5)
    xa, xb = _blocky(M, K, blk, 1, lo, hi), _blocky(N, K, blk, 2, lo, hi)
    if kind == "mxfp8":
        a, sfa = Q.quantize_mxfp8(xa)
        b, sfb = Q.quantize_mxfp8(xb)
        to_codes = lambda c: torch.from_numpy(c).cuda().view(torch.float8_e4m3fn)
        to_sf = lambda s: torch.from_numpy(s).cuda().view(torch.float8_e8m0fnu)
    else:
        if not hasattr(torch, "float4_e2m1fn_x2"):
            pytest.skip("this PyTorch has no float4_e2m1fn_x2")
        # a tensor scale of one: the UE4M3 block scales carry every magnitude
        a, sfa, _ = Q.quantize_nvfp4(xa, np.float32(1.0))
        b, sfb, _ = Q.quantize_nvfp4(xb, np.float32(1.0))
        to_codes = lambda c: torch.from_numpy(c).cuda().view(torch.float4_e2m1fn_x2)
        to_sf = lambda s: torch.from_numpy(s).cuda().view(torch.float8_e4m3fn)
    SFA, SFB = L.swizzle(sfa), L.swizzle(sfb)
    assert len(np.unique(sfa)) > 10 and len(np.unique(sfb)) > 10
    got = _scaled_mm(to_codes(a), to_codes(b), to_sf(SFA), to_sf(SFB))
    got = got.float().cpu().numpy().astype(np.float64)
    prob = dict(kind=kind, M=M, N=N, K=K, A=a, B=b, SFA=SFA, SFB=SFB, alpha=np.float32(1.0))
    P.assert_parity(got, prob, "bf16")
    # the same codes with the scale bytes of the other in-atom order: the oracle's result moves
    # far outside the bound, so agreement above is not an accident of uniform scales
    wrong = dict(prob, SFA=_other_order(sfa, M, K // blk), SFB=_other_order(sfb, N, K // blk))
    ref_w, _ = R.reference(kind, a, b, wrong["SFA"], wrong["SFB"], M, N, K, out="bf16")
    _, abs_sum = P.reference(prob, "bf16")
    tol = R.tolerance(ref_w, got, abs_sum, 1.0, False, "bf16")
    assert np.mean(np.abs(got - ref_w) > tol) > 0.5
