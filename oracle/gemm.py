"""Reference block-scaled GEMM: D = out_round(epi(alpha * A_hat @ B_hat^T)), in float64.

TEST INFRASTRUCTURE (part of the CPU oracle; see ``oracle/formats.py``).

What it follows:
* the operation and operand layouts of "Add Cutlass MxFp8 Block Scale Matrix
  Multiplication" (``MxFp8GemmSm100``: A row-major M x K, B given as N x K
  ("ColumnMajor" K x N), D row-major M x N, float accumulator, ``alpha_ptr`` in
  the epilogue; its test compares against ``get_ref_results`` on the dequantised
  operands);
* the NVFP4 entry ``runNvfp4Gemm<T, kEnableSilu, kEnableBias>`` of "[QST]
  Performance overhead: Frequent cuTensorMapEncodeTiled ...": a host float
  alpha, an optional bias and an optional SiLU, output type T.

The exact result of the method is a scaled dot product, so this is that
definition written out: every element and scale is decoded through the explicit
tables of ``formats``, the products are summed in float64 (``numpy.matmul`` is
the library primitive for the sum), then

    y = alpha * alpha_row[m] * alpha_col[n] * acc;  y = y + bias[n] (bias);
    y = y + beta * C[m, n] (C);  y = y / (1 + exp(-y)) (SiLU);
    D = y rounded to nearest even in the output type.

The per-row / per-column factors and the C term are the next-step epilogue of the
MXFP8 page's LinearCombination (alpha, beta and a C operand, there aliased to D),
with C kept separate; their order is this library's documented reading.

The scales are read from the swizzled buffers through ``layout.unswizzle`` so
that the byte map of the scale layout is exercised end to end.

NVFP4 output (the output half of the activation-quantiser step that the MXFP8
page's test performs before each GEMM): instead of rounding y to a 16-bit type,
each 16-column block of a row goes through the NVFP4 recipe of ``quantize`` with
a given global scale s, on y taken in float32 (the precision the recipe states);
``quantize_output_nvfp4``.
"""

import numpy as np

from . import formats as F
from . import layout as L
from .quantize import MX_BLOCK, NV_BLOCK, quantize_nvfp4, unpack_e2m1

MXFP8 = "mxfp8"
NVFP4 = "nvfp4"
BF16 = "bf16"
F16 = "f16"


def decode_operand(kind, codes, sf_buf, rows, K):
    """Element codes + swizzled scales -> float64 [rows, K] holding element * block scale."""
    if kind == MXFP8:
        codes = np.asarray(codes, dtype=np.uint8).reshape(rows, K)
        sf = L.unswizzle(sf_buf, rows, K // MX_BLOCK)
        return F.decode_e4m3(codes) * np.repeat(F.decode_ue8m0(sf), MX_BLOCK, axis=1)
    if kind == NVFP4:
        codes = unpack_e2m1(np.asarray(codes, dtype=np.uint8).reshape(rows, K // 2), K)
        sf = L.unswizzle(sf_buf, rows, K // NV_BLOCK)
        return F.decode_e2m1(codes) * np.repeat(F.decode_ue4m3(sf), NV_BLOCK, axis=1)
    raise ValueError(kind)


def effective_alpha(alpha, alpha_row=None, alpha_col=None):
    """alpha * alpha_row[m] * alpha_col[n] in float64 (a scalar, a column, a row or a matrix);
    every factor is a float32 value."""
    a = np.float64(np.float32(alpha))
    if alpha_row is not None:
        a = a * np.asarray(alpha_row, dtype=np.float32).astype(np.float64)[:, None]
    if alpha_col is not None:
        a = a * np.asarray(alpha_col, dtype=np.float32).astype(np.float64)[None, :]
    return a


def epilogue(acc, alpha, bias=None, silu=False, C=None, beta=0.0, alpha_row=None, alpha_col=None):
    """float64 accumulator -> float64 pre-rounding output (the factors, + bias[n], + beta C, SiLU).

    ``C`` holds the float64 values of the residual input (exact in the output type)."""
    y = effective_alpha(alpha, alpha_row, alpha_col) * np.asarray(acc, dtype=np.float64)
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :]
    if C is not None:
        y = y + np.float64(np.float32(beta)) * np.asarray(C, dtype=np.float64)
    if silu:
        with np.errstate(over="ignore"):
            y = y * (1.0 / (1.0 + np.exp(-y)))
    return y


def round_out(y, out):
    return F.round_to_bf16(y) if out == BF16 else F.round_to_f16(y)


def out_bits(v, out):
    return F.bf16_bits(v) if out == BF16 else F.f16_bits(v)


def out_from_bits(bits, out):
    return F.bf16_from_bits(bits) if out == BF16 else F.f16_from_bits(bits)


def ulp_out(v, out):
    return F.ulp_bf16(v) if out == BF16 else F.ulp_f16(v)


def reference(kind, A, B, SFA, SFB, M, N, K, alpha=1.0, bias=None, silu=False, out=BF16,
              rows=None, C=None, beta=0.0, alpha_row=None, alpha_col=None):
    """Reference D (float64 values, exactly representable in ``out``) and the pre-rounding y.

    ``bias`` is a float64 vector of the (already rounded) bias values, ``C`` the float64 M x N
    values of the residual input.  ``rows`` optionally selects a subset of output rows (for
    sampled checks of large problems); the result then has len(rows) rows.
    """
    Ahat = decode_operand(kind, A, SFA, M, K)
    if rows is not None:
        r = np.asarray(rows)
        Ahat = Ahat[r]
        C = None if C is None else np.asarray(C)[r]
        alpha_row = None if alpha_row is None else np.asarray(alpha_row)[r]
    Bhat = decode_operand(kind, B, SFB, N, K)
    acc = Ahat @ Bhat.T
    y = epilogue(acc, alpha, bias, silu, C, beta, alpha_row, alpha_col)
    return round_out(y, out), y


def abs_product_sum(kind, A, B, SFA, SFB, M, N, K, rows=None):
    """sum_k |a_hat[m,k] * b_hat[n,k]| in float64 (the scale of the accumulation error)."""
    Ahat = decode_operand(kind, A, SFA, M, K)
    if rows is not None:
        Ahat = Ahat[np.asarray(rows)]
    Bhat = decode_operand(kind, B, SFB, N, K)
    return np.abs(Ahat) @ np.abs(Bhat).T


def tolerance(ref, got, abs_sum, alpha, silu, out):
    """Per-element bound |alpha| * 2**-7 * sum|a b| (x 1.1 with SiLU) + 1 output ulp.

    ``alpha`` is the effective factor (a scalar, or ``effective_alpha`` with per-row /
    per-column factors).  The ulp is taken at the larger of |ref| and |got|, so that the
    rounding of either side to the output type is covered.
    """
    lip = 1.1 if silu else 1.0            # max |d silu / dy| = 1.0998...
    mag = np.maximum(np.abs(ref), np.abs(got))
    a = np.abs(np.asarray(alpha, dtype=np.float64)) if np.ndim(alpha) else abs(float(np.float32(alpha)))
    return a * 2.0 ** -7 * lip * abs_sum + ulp_out(mag, out)


def gemm_naive(kind, A, B, SFA, SFB, M, N, K, alpha=1.0, bias=None, silu=False, C=None, beta=0.0,
               alpha_row=None, alpha_col=None):
    """Triple loop in plain Python floats (float64): the same definition, no library sum."""
    Ahat = decode_operand(kind, A, SFA, M, K)
    Bhat = decode_operand(kind, B, SFB, N, K)
    acc = np.zeros((M, N), dtype=np.float64)
    for m in range(M):
        for n in range(N):
            t = 0.0
            for k in range(K):
                t += float(Ahat[m, k]) * float(Bhat[n, k])
            acc[m, n] = t
    return epilogue(acc, alpha, bias, silu, C, beta, alpha_row, alpha_col)


def quantize_output_nvfp4(y, s):
    """NVFP4 output of the epilogue: y (float64 [M, N], the values before output rounding) in
    float32, then per 16-column block of a row the NVFP4 recipe with global scale s.
    Returns (packed E2M1 codes uint8 [M, N/2], UE4M3 scale codes uint8 [M, N/16])."""
    codes, scales, _ = quantize_nvfp4(np.asarray(y, dtype=np.float64).astype(np.float32), np.float32(s))
    return codes, scales
