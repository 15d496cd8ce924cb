"""Quantisers: float32 matrices -> element codes + linear block scales.

TEST INFRASTRUCTURE (part of the CPU oracle; see ``oracle/formats.py``).

The pages call the MXFP8 quantiser (``pytorch_mxfp8_quantize`` in the test of
"Add Cutlass MxFp8 Block Scale Matrix Multiplication", block size 32) but print
no body, and say nothing of the NVFP4 one beyond the format name.  The steps
below are the plainest readings of the stated recipes:

MXFP8, per (row, 32-element K-block):
  1. amax = max |x| over the block (exact in float32);
  2. e = the smallest integer with amax <= 448 * 2**e, i.e. ceil(log2(amax / 448))
     taken exactly, clamped to [-127, 127]; the scale code is e + 127 (UE8M0);
  3. each element becomes E4M3(x * 2**-e), the product rounded in float32 and the
     code rounded to nearest even with saturation.

NVFP4, per tensor and per (row, 16-element K-block), every step one float32
operation rounded to nearest even:
  1. s = amax_tensor / 2688 (2688 = 448 * 6, the largest UE4M3 times the largest E2M1);
  2. d = 6 * s;  t = amax_block / d (0 when d == 0);  scale code = UE4M3(t);
  3. den = value(scale) * s;  q = x / den (0 when den == 0);  element = E2M1(q);
  4. the GEMM's global factor is alpha = s_A * s_B.
"""

import math

import numpy as np

from . import formats as F

MX_BLOCK = 32
NV_BLOCK = 16


def mx_scale_exponent(amax):
    """Smallest integer e with amax <= 448 * 2**e, clamped to [-127, 127] (amax >= 0, finite)."""
    amax = float(amax)
    if amax == 0.0:
        return -127
    e = math.ceil(math.log2(amax / F.E4M3_MAX))
    # log2 in floating point can be off by one near powers of two: settle it exactly.
    while amax > math.ldexp(F.E4M3_MAX, e):
        e += 1
    while amax <= math.ldexp(F.E4M3_MAX, e - 1):
        e -= 1
    return max(-127, min(127, e))


def mx_scale_exponents(amax):
    """Array form of :func:`mx_scale_exponent` (same steps, element-wise)."""
    a = np.asarray(amax, dtype=np.float64)
    pos = a > 0
    with np.errstate(divide="ignore"):
        e = np.where(pos, np.ceil(np.log2(np.where(pos, a, 1.0) / F.E4M3_MAX)), -127).astype(np.int64)
    while True:                                   # exact settle, as in the scalar form
        up = pos & (a > np.ldexp(F.E4M3_MAX, e))
        if not up.any():
            break
        e = e + up
    while True:
        down = pos & (a <= np.ldexp(F.E4M3_MAX, e - 1))
        if not down.any():
            break
        e = e - down
    return np.clip(e, -127, 127)


def quantize_mxfp8(x):
    """float32 [rows, K] -> (E4M3 codes uint8 [rows, K], UE8M0 scales uint8 [rows, K/32])."""
    x = np.asarray(x, dtype=np.float32)
    rows, K = x.shape
    if K % MX_BLOCK:
        raise ValueError("K must be a multiple of 32")
    nb = K // MX_BLOCK
    xb = x.reshape(rows, nb, MX_BLOCK)
    amax = np.max(np.abs(xb), axis=2)                                   # float32, exact
    e = mx_scale_exponents(amax)
    inv_scale = np.ldexp(np.float32(1.0), (-e).astype(np.int32)).astype(np.float32)   # 2**-e, exact in fp32
    q = (xb * inv_scale[:, :, None]).astype(np.float32)                  # float32 product, RNE
    codes = F.encode_e4m3(q).reshape(rows, K)
    scales = (e + 127).astype(np.uint8)
    return codes, scales


def nvfp4_global_scale(x):
    """s = amax(|x|) / 2688 in float32."""
    amax = np.float32(np.max(np.abs(np.asarray(x, dtype=np.float32)))) if np.size(x) else np.float32(0)
    return np.float32(amax / np.float32(2688.0))


def quantize_nvfp4(x, s=None):
    """float32 [rows, K] -> (packed E2M1 uint8 [rows, K/2], UE4M3 scales uint8 [rows, K/16], s float32).

    Element 2j of a row sits in the low nibble of byte j, element 2j+1 in the high nibble.
    """
    x = np.asarray(x, dtype=np.float32)
    rows, K = x.shape
    if K % NV_BLOCK:
        raise ValueError("K must be a multiple of 16")
    if s is None:
        s = nvfp4_global_scale(x)
    s = np.float32(s)
    nb = K // NV_BLOCK
    xb = x.reshape(rows, nb, NV_BLOCK)
    amax_b = np.max(np.abs(xb), axis=2).astype(np.float32)
    d = np.float32(np.float32(6.0) * s)
    if d == 0:
        t = np.zeros_like(amax_b)
    else:
        t = (amax_b / d).astype(np.float32)
    sc = F.encode_ue4m3(t)                                               # uint8 [rows, nb]
    den = (F.decode_ue4m3(sc).astype(np.float32) * s).astype(np.float32)  # exact decode, fp32 product
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(den[:, :, None] != 0, xb / den[:, :, None], np.float32(0)).astype(np.float32)
    codes = F.encode_e2m1(q).reshape(rows, K) & 0xF
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, sc.astype(np.uint8), s


def quantize_mxfp8_bf16(bits):
    """BF16 bit patterns [rows, K] -> quantize_mxfp8 of their values (every BF16 value is a
    float32, so the widening is exact and the recipe is the float32 one unchanged)."""
    return quantize_mxfp8(F.decode_bf16(bits).astype(np.float32))


def quantize_nvfp4_bf16(bits, s=None):
    """BF16 bit patterns [rows, K] -> quantize_nvfp4 of their values (see quantize_mxfp8_bf16)."""
    return quantize_nvfp4(F.decode_bf16(bits).astype(np.float32), s)


def unpack_e2m1(packed, K):
    """uint8 [rows, K/2] -> E2M1 codes uint8 [rows, K] (low nibble first)."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows = packed.shape[0]
    out = np.empty((rows, K), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out
