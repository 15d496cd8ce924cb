"""Pins of the oracle's quantisers: exact rational invariants and brute force.

MXFP8: the scale exponent is the least e with amax <= 448 * 2**e (checked with
exact fractions), and every element is the nearest E4M3 value of x / 2**e
(exhaustive search).  NVFP4: hand-chosen inputs where every float32 step is
exact, so the codes are known in closed form; the general case is checked
element by element against an exhaustive nearest-value search of x / den; and
elements within a few ulps of every E2M1 threshold against E2M1(RN(x / den))
computed with exact rationals (no float32 division: an oracle that multiplied by
a rounded reciprocal instead fails this pin and passes the brute-force one); block
amaxes near every E4M3 midpoint likewise for the scale step.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import formats as F
from oracle import quantize as Q
from fp4_gemm_blackwell_gb300 import synth


def _nearest_brute(v, table, maxv, ncodes):
    mag = min(abs(v), maxv)
    best = None
    for c in range(ncodes):
        t = table[c]
        if np.isnan(t) or t < 0 or (t == 0 and np.signbit(t)):
            continue
        d = abs(Fraction(mag) - Fraction(t))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def test_mx_scale_exponent_is_minimal_exact():
    rng = np.random.default_rng(0)
    amax = np.concatenate([np.abs(rng.normal(0, 1, 500)) * 10.0 ** rng.integers(-30, 30, 500),
                           [448.0, 448.0 * 2 ** 5, 448.0 * 2 ** -9, np.nextafter(448.0, 1e9, dtype=np.float32),
                            np.nextafter(448.0, 0, dtype=np.float32), 1.0, 3.4e38]]).astype(np.float32)
    for a in amax:
        e = Q.mx_scale_exponent(a)
        fa = Fraction(float(a))
        assert fa <= 448 * Fraction(2) ** e
        assert fa > 448 * Fraction(2) ** (e - 1)
    vec = Q.mx_scale_exponents(amax.astype(np.float64))
    assert list(vec) == [Q.mx_scale_exponent(a) for a in amax]
    # boundaries: amax exactly 448 * 2^k gives e = k; one float32 ulp above gives k + 1
    assert Q.mx_scale_exponent(448.0) == 0
    assert Q.mx_scale_exponent(448.0 * 2 ** 3) == 3
    assert Q.mx_scale_exponent(float(np.nextafter(np.float32(448.0), np.float32(1e9)))) == 1
    assert Q.mx_scale_exponent(0.0) == -127
    assert Q.mx_scale_exponent(1e-45) == -127                         # clamp


def test_mx_quantiser_against_brute_force():
    x = synth.normal(4, 96, seed=5) * np.float32(3.0)
    x[1, :32] *= np.float32(1e-6)                                      # a small block
    x[2, 32:64] = 0.0                                                  # an all-zero block
    codes, scales = Q.quantize_mxfp8(x)
    assert codes.shape == (4, 96) and scales.shape == (4, 3)
    for r in range(4):
        for b in range(3):
            blk = x[r, 32 * b:32 * b + 32].astype(np.float64)
            e = int(scales[r, b]) - 127
            amax = np.max(np.abs(blk))
            if amax == 0:
                assert e == -127
                assert np.all(codes[r, 32 * b:32 * b + 32] == 0)
                continue
            assert Fraction(amax) <= 448 * Fraction(2) ** e < 2 * Fraction(amax)
            for j in range(32):
                q = blk[j] * 2.0 ** -e
                want = _nearest_brute(q, F.E4M3_VALUES, 448.0, 127)
                if np.signbit(q):
                    want |= 0x80
                assert codes[r, 32 * b + j] == want


def test_mx_block_max_maps_inside_range():
    x = synth.normal(64, 256, seed=9) * np.float32(1000.0)
    codes, scales = Q.quantize_mxfp8(x)
    dec = F.decode_e4m3(codes).reshape(64, 8, 32)
    assert np.all(np.abs(dec) <= 448.0)
    # each block's largest magnitude lands in the top binade [256, 448]
    assert np.all(np.max(np.abs(dec), axis=2) >= 224.0)


def test_nv_closed_form_case():
    # amax_tensor = 2688 -> s = 1 exactly; a block with amax 6 -> t = 1 -> scale 1.0 (code 0x38);
    # den = 1, so every element is E2M1(x) directly, ties included.
    row0 = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0, 0.1, 0.3, 4.4, -6.0, 1.0],
                    dtype=np.float32)
    row1 = np.zeros(16, dtype=np.float32)
    row1[0] = 2688.0
    x = np.stack([row0, row1])
    packed, sc, s = Q.quantize_nvfp4(x)
    assert s == np.float32(1.0)
    assert sc[0, 0] == 0x38
    assert sc[1, 0] == 0x7E                                           # 2688 / 6 = 448 -> max UE4M3
    codes = Q.unpack_e2m1(packed, 16)[0]
    vals = F.decode_e2m1(codes)
    assert list(vals) == [6.0, 0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -0.0, -1.0, -4.0, 0.0, 0.5, 4.0, -6.0, 1.0]
    # nibble order: element 0 in the low nibble
    assert packed[0, 0] & 0xF == codes[0] and packed[0, 0] >> 4 == codes[1]


def test_nv_quantiser_against_brute_force():
    x = synth.normal_rowscaled(6, 64, seed=4)
    packed, sc, s = Q.quantize_nvfp4(x)
    assert s == np.float32(np.float32(np.max(np.abs(x))) / np.float32(2688.0))
    codes = Q.unpack_e2m1(packed, 64)
    d = np.float32(np.float32(6.0) * s)
    for r in range(6):
        for b in range(4):
            blk = x[r, 16 * b:16 * b + 16]
            t = np.float32(np.float32(np.max(np.abs(blk))) / d)
            want_sc = _nearest_brute(float(t), F.E4M3_VALUES, 448.0, 127)
            assert sc[r, b] == want_sc
            den = np.float32(np.float32(F.E4M3_VALUES[want_sc]) * s)
            for j in range(16):
                q = float(np.float32(blk[j] / den))
                want = _nearest_brute(q, F.E2M1_VALUES, 6.0, 8) | (0x8 if np.signbit(q) else 0)
                assert codes[r, 16 * b + j] == want


def _rn_float32(q):
    """The float32 nearest to the non-negative rational q, ties to the even significand (normal
    and subnormal range; these tests stay far from overflow)."""
    if q == 0:
        return Fraction(0)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    e = max(e, -126)                                  # below 2^-126 the spacing stays 2^-149
    scaled = q * Fraction(2) ** (23 - e)              # significand in units of the last place
    n, rem = divmod(scaled.numerator, scaled.denominator)
    twice = 2 * rem
    if twice > scaled.denominator or (twice == scaled.denominator and n % 2 == 1):
        n += 1
    return Fraction(n) * Fraction(2) ** (e - 23)


def _e2m1_code_exact(v):
    """E2M1 code of the float32 value v (a Fraction, any sign): the nearest magnitude of the
    value set, ties to the even code, saturating at 6, sign bit 0x8."""
    mag = min(abs(v), Fraction(6))
    vals = [Fraction(x) for x in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    best = min(range(8), key=lambda c: (abs(mag - vals[c]), c % 2))
    return best | (0x8 if v < 0 else 0)


def test_nv_elements_near_thresholds_match_exact_rationals():
    # Dividends RN(T * den) and up to 4 float32 ulps either side of every E2M1 rounding threshold
    # T, for block scales den = value(code) * s with s = amax / 2688 of a tensor whose amax has a
    # long significand: the oracle's element codes against E2M1(RN(x / den)) computed with exact
    # rationals, where numpy's float32 division is not used at all.
    rng = np.random.default_rng(11)
    thresholds = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for amax in (np.float32(10.3125), np.float32(2688.0), np.float32(rng.uniform(1, 100))):
        s = np.float32(amax / np.float32(2688.0))
        for code in (0x30, 0x35, 0x3B, 0x41, 0x4E, 0x57):
            den = np.float32(np.float32(F.E4M3_VALUES[code]) * s)
            cand = []
            for T in thresholds:
                base = np.float32(np.float32(T) * den)
                for k in range(-4, 5):
                    v = np.float32(base)
                    step = np.float32(np.inf) if k > 0 else np.float32(0)
                    for _ in range(abs(k)):
                        v = np.nextafter(v, step)
                    cand.append(v)
            cand = np.array(cand, dtype=np.float32)
            cand[1::2] *= -1
            for i in range(0, len(cand), 15):
                blk = np.zeros(16, dtype=np.float32)
                blk[0] = np.float32(np.float32(6.0) * den)     # block amax: its scale is `code`
                chunk = cand[i:i + 15]
                blk[1:1 + len(chunk)] = chunk
                x = np.stack([blk, np.r_[amax, np.zeros(15, dtype=np.float32)].astype(np.float32)])
                packed, sc, s_out = Q.quantize_nvfp4(x)
                assert s_out == s and sc[0, 0] == code
                codes = Q.unpack_e2m1(packed, 16)[0]
                den_q = Fraction(float(den))
                for j in range(16):
                    q = _rn_float32(abs(Fraction(float(blk[j])) / den_q))
                    want = _e2m1_code_exact(-q if np.signbit(blk[j]) else q)
                    if q == 0 and np.signbit(blk[j]):
                        want = 0x8
                    assert codes[j] == want, (float(blk[j]), float(den), codes[j], want)


def test_nv_block_scales_near_midpoints_match_exact_rationals():
    # Block amaxes RN(m * d) and up to 3 float32 ulps either side of every midpoint m between two
    # neighbouring E4M3 values (and past the largest), for given global scales with long
    # significands: the oracle's scale codes against UE4M3(RN(amax / d)) computed with exact
    # rationals (no float32 division).
    pos = [c for c in range(0x7F) if np.isfinite(F.E4M3_VALUES[c])]
    vals = [Fraction(float(F.E4M3_VALUES[c])) for c in pos]
    mids = [(vals[i] + vals[i + 1]) / 2 for i in range(len(vals) - 1)] + [Fraction(464)]
    for s in (np.float32(np.float32(10.3125) / np.float32(2688.0)), np.float32(0.0123456789),
              np.float32(3.3333333)):
        d = np.float32(np.float32(6.0) * s)
        d_q = Fraction(float(d))
        amaxes = []
        for m in mids:
            base = np.float32(float(m * d_q))
            for k in range(-3, 4):
                v = base
                for _ in range(abs(k)):
                    v = np.nextafter(v, np.float32(np.inf) if k > 0 else np.float32(0))
                amaxes.append(v)
        x = np.zeros((len(amaxes), 16), dtype=np.float32)
        x[:, 0] = amaxes
        _, sc, s_out = Q.quantize_nvfp4(x, s)
        assert s_out == s
        for r, a in enumerate(amaxes):
            t = _rn_float32(Fraction(float(a)) / d_q)
            mag = min(t, Fraction(448))
            want = pos[min(range(len(pos)), key=lambda i: (abs(mag - vals[i]), pos[i] % 2))]
            assert sc[r, 0] == want, (float(a), float(d), sc[r, 0], want)


def test_nv_tensor_amax_block_gets_max_scale():
    x = synth.normal_rowscaled(32, 128, seed=8)
    packed, sc, s = Q.quantize_nvfp4(x)
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sc[r, c // 16] == 0x7E


def test_nv_all_zero_tensor():
    packed, sc, s = Q.quantize_nvfp4(np.zeros((4, 32), dtype=np.float32))
    assert s == 0 and not packed.any() and not sc.any()


@pytest.mark.parametrize("kind", ["mx", "nv"])
def test_dequantised_error_is_within_half_step(kind):
    x = synth.normal(16, 128, seed=21)
    if kind == "mx":
        codes, scales = Q.quantize_mxfp8(x)
        deq = F.decode_e4m3(codes) * np.repeat(F.decode_ue8m0(scales), 32, axis=1)
        # E4M3 relative step 2^-3 in normal range: |err| <= 2^-4 * |x| + tiny subnormal step
        step = np.repeat(F.decode_ue8m0(scales), 32, axis=1) * 2.0 ** -9
        assert np.all(np.abs(deq - x) <= np.abs(x) * 2.0 ** -4 + step / 2 + 1e-30)
    else:
        packed, sc, s = Q.quantize_nvfp4(x)
        codes = Q.unpack_e2m1(packed, 128)
        scale = np.repeat(F.decode_ue4m3(sc), 16, axis=1) * float(s)
        deq = F.decode_e2m1(codes) * scale
        # E2M1 spacing is at most 2 (between 4 and 6), so |err| <= 1 * block scale, plus scale rounding
        assert np.all(np.abs(deq - x) <= 1.0 * scale * 1.07 + 1e-30)


def test_bf16_decode_exhaustive():
    # every 16-bit pattern, against the float32 whose upper half it is (a reinterpretation by
    # numpy, not the oracle's field decode): equal values, NaN exactly where the pattern is NaN
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = F.decode_bf16(bits)
    want = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # hand-checked patterns: 1, -2, the largest finite, the smallest subnormal, +-inf, -0
    assert F.decode_bf16(np.array([0x3F80, 0xC000, 0x7F7F, 0x0001, 0x7F80, 0xFF80], np.uint16)).tolist() == [
        1.0, -2.0, float.fromhex("0x1.fep127"), 2.0 ** -133, float("inf"), float("-inf")]
    z = F.decode_bf16(np.array([0x8000], np.uint16))[0]
    assert z == 0.0 and np.signbit(z)


def test_bf16_quantisers_quantise_the_widened_values():
    # the BF16 entry points apply the float32 recipe to the exactly widened values
    x = synth.normal_rowscaled(8, 96, seed=3)
    bits = synth.as_bf16_bits(x)
    wide = (bits.astype(np.uint32) << 16).view(np.float32)
    c0, s0 = Q.quantize_mxfp8_bf16(bits)
    c1, s1 = Q.quantize_mxfp8(wide)
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
    p0, t0, g0 = Q.quantize_nvfp4_bf16(bits)
    p1, t1, g1 = Q.quantize_nvfp4(wide)
    assert np.array_equal(p0, p1) and np.array_equal(t0, t1) and g0 == g1


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_row_chunked_quantisation_equals_whole_matrix(kind):
    # the large GPU parity cases quantise their operands in row chunks in worker processes:
    # the bytes must be those of one oracle call on the whole matrix (NVFP4: the chunks take
    # the whole matrix's tensor scale); rows = 300 gives chunks of unequal size
    import oracle_pool
    from oracle import layout as L
    x = synth.normal_rowscaled(300, 256, seed=9)
    x[17] *= 40.0                        # the tensor amax sits in one chunk only
    if kind == "mxfp8":
        want_c, want_s = Q.quantize_mxfp8(x)
        want_g = None
    else:
        want_c, want_s, want_g = Q.quantize_nvfp4(x)
    for parts in (1, 7):
        c, s, g = oracle_pool.quantize_rows(kind, x, parts=parts)
        assert np.array_equal(c, want_c) and np.array_equal(s, want_s) and g == want_g
    pool = oracle_pool.spawn_pool(2)
    try:
        c, sw, g = oracle_pool.operand(kind, x, pool)
    finally:
        pool.close()
        pool.join()
    assert np.array_equal(c, want_c) and np.array_equal(sw, L.swizzle(want_s)) and g == want_g
