"""Pins of the oracle's codecs and output rounding against facts from outside the oracle.

* the OCP MX v1.0 format facts in tests/golden/format_values.txt;
* PyTorch's own float8_e4m3fn / float8_e8m0fnu decoders (a library routine);
* PyTorch's float32 -> float8_e4m3fn cast, which rounds to nearest even below
  the overflow threshold (it returns NaN rather than saturating above it);
* numpy's float64 -> float16 cast and PyTorch's float32 -> bfloat16 cast, both
  correctly rounded to nearest even;
* exhaustive nearest-value search over the code tables.
"""

import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "format_values.txt")


def _golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, *v = line.split()
        out[k] = v
    return out


G = _golden()


def _num(s):
    return int(s, 16) if s.startswith("0x") else float(s)


def test_e4m3_table_matches_golden_facts():
    v = F.E4M3_VALUES
    assert v[_num(G["e4m3_max_finite_code"][0])] == _num(G["e4m3_max_finite"][0])
    assert np.nanmax(v) == 448.0 and np.nanmin(v) == -448.0
    nan_codes = sorted(int(c) for c in np.flatnonzero(np.isnan(v)))
    assert nan_codes == [_num(c) for c in G["e4m3_nan_codes"]]
    pos = v[:0x7F]
    assert pos[1] == _num(G["e4m3_min_subnormal"][0])
    assert pos[8] == _num(G["e4m3_min_normal"][0])
    assert v[_num(G["e4m3_one_code"][0])] == 1.0
    assert np.all(np.diff(pos) > 0)                           # monotone in the code
    assert np.array_equal(v[0x80:0xFF], -pos)                 # sign-magnitude


def test_e4m3_table_matches_torch_decoder():
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(t), np.isnan(F.E4M3_VALUES))
    ok = ~np.isnan(t)
    assert np.array_equal(t[ok], F.E4M3_VALUES[ok])
    assert np.array_equal(np.signbit(t[ok]), np.signbit(F.E4M3_VALUES[ok]))


def test_e2m1_table_matches_golden_values():
    want = [float(x) for x in G["e2m1_positive_values"]]
    assert list(F.E2M1_VALUES[:8]) == want
    assert list(F.E2M1_VALUES[8:]) == [-x for x in want]
    assert F.E2M1_MAX == _num(G["e2m1_max"][0])


def test_ue8m0_table_matches_torch_decoder_and_golden():
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.isnan(t[255]) and np.isnan(F.UE8M0_VALUES[255])
    assert np.array_equal(t[:255], F.UE8M0_VALUES[:255])
    assert F.UE8M0_VALUES[int(_num(G["ue8m0_bias"][0]))] == 1.0
    assert F.UE8M0_VALUES[0] == _num(G["ue8m0_min"][0])


def test_ue4m3_is_unsigned_e4m3():
    assert np.array_equal(F.UE4M3_VALUES[:127], F.E4M3_VALUES[:127])
    assert np.all(np.isnan(F.UE4M3_VALUES[128:]))


@pytest.mark.parametrize("name", ["e4m3", "e2m1"])
def test_round_trip_every_code(name):
    if name == "e4m3":
        codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
        assert np.array_equal(F.encode_e4m3(F.decode_e4m3(codes)), codes)
    else:
        codes = np.arange(16, dtype=np.uint8)
        assert np.array_equal(F.encode_e2m1(F.decode_e2m1(codes)), codes)


def _brute_nearest(x, table, codes, maxv):
    """Nearest finite table value by exhaustive search; ties -> even code; saturate."""
    out = []
    for xv in x:
        mag = min(abs(xv), maxv)
        best = None
        for c, v in zip(codes, table):
            if np.isnan(v) or v < 0 or (v == 0 and np.signbit(v)):
                continue
            d = abs(mag - v)
            if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
                best = (d, c)
        c = best[1]
        out.append(c | ((0x80 if len(table) == 256 else 0x8) if np.signbit(xv) else 0))
    return np.array(out, dtype=np.uint8)


def test_encoders_match_exhaustive_search_and_ties():
    rng = np.random.default_rng(7)
    pos = F.E4M3_VALUES[:0x7F]
    mids = (pos[1:] + pos[:-1]) / 2                                  # every tie
    x = np.concatenate([mids, -mids, rng.normal(0, 50, 2000), rng.normal(0, 0.01, 500),
                        [1e6, -1e6, 448.0, 464.0, 463.9, 0.0, -0.0]]).astype(np.float32)
    got = F.encode_e4m3(x)
    want = _brute_nearest(x.astype(np.float64), F.E4M3_VALUES, range(256), 448.0)
    assert np.array_equal(got, want)

    p2 = F.E2M1_VALUES[:8]
    mids2 = (p2[1:] + p2[:-1]) / 2
    x2 = np.concatenate([mids2, -mids2, rng.normal(0, 3, 2000), [7.0, -100.0, 0.25, 0.2499]]).astype(np.float32)
    got2 = F.encode_e2m1(x2)
    want2 = _brute_nearest(x2.astype(np.float64), F.E2M1_VALUES, range(16), 6.0)
    assert np.array_equal(got2, want2)
    # spelled-out ties of E2M1: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    assert list(F.decode_e2m1(F.encode_e2m1(ties))) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_e4m3_encoder_matches_torch_cast_below_overflow():
    rng = np.random.default_rng(3)
    pos = F.E4M3_VALUES[:0x7F]
    mids = (pos[1:] + pos[:-1]) / 2
    x = np.concatenate([mids, -mids, rng.uniform(-463, 463, 20000),
                        rng.normal(0, 1e-3, 2000)]).astype(np.float32)
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.encode_e4m3(x), t)


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(11)
    y = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-5, 2000), rng.normal(0, 3e4, 2000),
                        [65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]])
    ours = F.round_to_f16(y)
    with np.errstate(over="ignore"):
        lib = y.astype(np.float16).astype(np.float64)
    assert np.array_equal(ours, lib)


def test_bf16_rounding_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(12)
    y32 = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-30, 1000),
                          rng.normal(0, 1e37, 1000)]).astype(np.float32)
    # exact ties: bf16 value + half a bf16 quantum, both parities
    base = torch.from_numpy(rng.normal(0, 1, 1000).astype(np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
    ties = (base.astype(np.float64) + F.ulp_bf16(base) / 2).astype(np.float32)
    y32 = np.concatenate([y32, ties, np.float32([3.3895314e38, -3.3895314e38])])
    ours = F.round_to_bf16(y32.astype(np.float64))
    lib = torch.from_numpy(y32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, lib)
    assert np.array_equal(F.bf16_from_bits(F.bf16_bits(ours)), ours)
