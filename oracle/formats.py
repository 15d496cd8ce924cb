"""Element and scale codecs of the block-scaled formats, in float64.

TEST INFRASTRUCTURE. This package is the slow, obviously-correct CPU oracle of
the block-scaled GEMM. Only the tests, the smoke check and the benchmark's CPU
baseline may import it; the product path never does.

Formats (the pages name them, the OCP Microscaling Formats (MX) v1.0
specification defines them):

* E4M3 -- the MXFP8 element ("Add Cutlass MxFp8 Block Scale Matrix
  Multiplication", ``MxFp8GemmSm100``: ``mx_float8_t<float_e4m3_t>``; validation
  step "Validate dtypes (Float8_e4m3fn, ...)").  Bits s|eeee|mmm, bias 7, no
  infinities, S.1111.111 is NaN, largest finite 448.
* UE8M0 -- the MXFP8 block scale (same page, ``ElementSFA = float_ue8m0_t``;
  dtype ``Float8_e8m0fnu``).  Eight exponent bits, value 2**(e-127), 0xFF NaN.
* E2M1 -- the NVFP4 element ("[QST] Performance overhead ...", the
  ``KernelTmaWarpSpecialized1SmNvf4Sm100`` mainloop).  Bits s|ee|m, bias 1,
  values +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}.  Two per byte.
* UE4M3 -- the NVFP4 block scale: an E4M3 with the sign bit zero.

Every table below is built from the bit fields, not by casting through a
hardware type.
"""

import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def _e4m3_value(code):
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** -6          # subnormal: 0.mmm * 2^(1-7)
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def _e2m1_value(code):
    s = (code >> 3) & 1
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        mag = m * 0.5                         # subnormal: 0.m * 2^(1-1)
    else:
        mag = (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


def _ue8m0_value(code):
    if code == 0xFF:
        return float("nan")
    return 2.0 ** (code - 127)


# Decode tables, indexed by the raw code.
E4M3_VALUES = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
E2M1_VALUES = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
UE8M0_VALUES = np.array([_ue8m0_value(c) for c in range(256)], dtype=np.float64)
# UE4M3 is only defined for sign-bit-clear bytes; a set sign bit decodes to NaN
# so that a misplaced byte cannot pass unnoticed.
UE4M3_VALUES = np.array([E4M3_VALUES[c] if c < 128 else float("nan") for c in range(256)],
                        dtype=np.float64)


def decode_e4m3(codes):
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def decode_e2m1(codes):
    return E2M1_VALUES[np.asarray(codes, dtype=np.uint8) & 0xF]


def decode_ue8m0(codes):
    return UE8M0_VALUES[np.asarray(codes, dtype=np.uint8)]


def decode_ue4m3(codes):
    return UE4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def _nearest_code(x, pos_codes, pos_values, max_value, sign_bit):
    """Round-to-nearest-even with saturation onto a sign-magnitude code set.

    ``pos_values`` are the finite non-negative values in increasing order and
    ``pos_codes`` their codes (increasing too, so an even code is an even
    mantissa LSB).  A magnitude above the largest finite value saturates to it
    (the ``satfinite`` behaviour); a tie picks the code whose last bit is 0.
    The sign bit is copied from the input, so -0.0 keeps it.
    """
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(np.abs(x), max_value)
    hi = np.searchsorted(pos_values, mag, side="left")          # first value >= mag
    hi = np.minimum(hi, len(pos_values) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - pos_values[lo]
    d_hi = pos_values[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((pos_codes[hi] & 1) == 0))
    exact = pos_values[hi] == mag
    code = np.where(exact | pick_hi, pos_codes[hi], pos_codes[lo]).astype(np.uint8)
    neg = np.signbit(x)
    return np.where(neg, code | sign_bit, code).astype(np.uint8)


_E4M3_POS_CODES = np.arange(0, 0x7F, dtype=np.int64)            # 0x00..0x7E finite
_E4M3_POS_VALUES = E4M3_VALUES[_E4M3_POS_CODES]
_E2M1_POS_CODES = np.arange(0, 8, dtype=np.int64)
_E2M1_POS_VALUES = E2M1_VALUES[_E2M1_POS_CODES]


def encode_e4m3(x):
    """float -> E4M3 code, round to nearest even, saturating at +-448."""
    return _nearest_code(x, _E4M3_POS_CODES, _E4M3_POS_VALUES, E4M3_MAX, 0x80)


def encode_e2m1(x):
    """float -> E2M1 code (low nibble), round to nearest even, saturating at +-6."""
    return _nearest_code(x, _E2M1_POS_CODES, _E2M1_POS_VALUES, E2M1_MAX, 0x8)


def encode_ue4m3(x):
    """non-negative float -> UE4M3 code (E4M3 with the sign bit clear)."""
    x = np.asarray(x, dtype=np.float64)
    if np.any(x < 0):
        raise ValueError("UE4M3 takes non-negative inputs")
    return encode_e4m3(np.abs(x)) & 0x7F


# ---- output rounding: float64 -> IEEE half / bfloat16, round to nearest even ----

def _round_binary(y, mant_bits, emin, emax):
    """Round float64 values to a binary format with ``mant_bits`` fraction bits,
    normal exponents in [emin, emax] and gradual underflow; overflow -> inf.

    The quantum of a value with floor(log2|y|) = q is 2**(max(q, emin) - mant_bits);
    dividing by a power of two is exact in float64 and ``np.rint`` rounds
    half to even.
    """
    y = np.asarray(y, dtype=np.float64)
    out = np.array(y, copy=True)
    a = np.abs(y)
    finite_nz = np.isfinite(a) & (a > 0)
    _, E = np.frexp(np.where(finite_nz, a, 1.0))                 # a = f * 2^E, f in [0.5, 1)
    q = np.maximum(E - 1, emin)
    quantum = np.ldexp(1.0, q - mant_bits)
    r = np.rint(np.where(finite_nz, a, 0.0) / quantum) * quantum
    largest = (2.0 - 2.0 ** -mant_bits) * 2.0 ** emax
    r = np.where(r > largest, np.inf, r)
    out = np.where(finite_nz, np.copysign(r, y), y)
    return out


def round_to_bf16(y):
    """float64 -> float64 holding the nearest bfloat16 (8 exponent bits, 7 fraction bits)."""
    return _round_binary(y, 7, -126, 127)


def round_to_f16(y):
    """float64 -> float64 holding the nearest IEEE binary16 (5 exponent bits, 10 fraction bits)."""
    return _round_binary(y, 10, -14, 15)


def bf16_bits(v):
    """Exact bfloat16 value (as float64) -> its 16-bit pattern."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)      # exact: a bf16 value is an fp32 value
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def f16_bits(v):
    """Exact binary16 value (as float64) -> its 16-bit pattern."""
    return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_from_bits(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def decode_bf16(bits):
    """BF16 bit patterns -> float64 values from the bit fields s|eeeeeeee|fffffff (bias 127):
    e = 0 gives (f/128) 2^-126, e = 255 gives +-inf (f = 0) or NaN, otherwise (1 + f/128) 2^(e-127).
    The input of the BF16 quantiser (each value is then an exact float32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 7) & 0xFF
    f = (b & 0x7F).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(f / 128.0, -126), np.ldexp(1.0 + f / 128.0, np.clip(e, 1, 254) - 127))
    mag = np.where(e == 255, np.where(f == 0, np.inf, np.nan), mag)
    return s * mag


def f16_from_bits(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def ulp_bf16(v):
    """Spacing of bfloat16 values at |v| (the quantum of the binade holding v)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    q = np.where(a > 0, np.maximum(E - 1, -126), -126)
    return np.ldexp(1.0, q - 7)


def ulp_f16(v):
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    q = np.where(a > 0, np.maximum(E - 1, -14), -14)
    return np.ldexp(1.0, q - 10)
