"""Pins of the oracle GEMM and epilogue.

* exact rational brute force on 4 x 4 x 32 (MXFP8) and 4 x 4 x 32 (NVFP4):
  elements decoded by PyTorch's float8 decoders / the E2M1 value list, scales
  read from the LINEAR (unswizzled) scale matrix, sums in Fractions;
* one-hot rows select single decoded elements times their scales;
* constant matrices give K * a * b * scales exactly;
* A and B are not interchangeable (D[m, n] pairs row m of A with row n of B);
* the triple loop and the library sum agree;
* the epilogue: bias is per output column, SiLU(0) = 0 and SiLU(y) -> y for large y;
  the residual and per-row / per-column factors: a zero operand leaves bias + beta C exactly,
  one-hot rows pick alpha * alpha_row[m] * alpha_col[n] times one decoded element, and C / the
  row factor follow their row through a sampled-rows evaluation.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as R
from oracle import layout as L
from oracle import quantize as Q
from fp4_gemm_blackwell_gb300 import synth

E2M1_LIST = [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def _torch_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_e8m0(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e8m0fnu).to(torch.float64).numpy()


def _e2m1_from_list(code):
    v = E2M1_LIST[code & 7]
    return -v if code & 8 else v


def _mx_operands(rows, K, seed, scale_spread=6):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C                              # no NaN codes
    sf = rng.integers(127 - scale_spread, 127 + scale_spread + 1, size=(rows, K // 32), dtype=np.uint8)
    return codes, sf


def _nv_operands(rows, K, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(rows, K), dtype=np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sf = rng.integers(1, 127, size=(rows, K // 16), dtype=np.uint8)
    return codes, packed, sf


def test_mx_bruteforce_4x4x32_exact():
    M = N = 4
    K = 32 * 2
    a, sfa = _mx_operands(M, K, 1)
    b, sfb = _mx_operands(N, K, 2)
    ad, bd = _torch_e4m3(a), _torch_e4m3(b)
    sa, sb = _torch_e8m0(sfa), _torch_e8m0(sfb)
    got, _ = R.reference(R.MXFP8, a, b, L.swizzle(sfa), L.swizzle(sfb), M, N, K, out=R.BF16)
    y = R.reference(R.MXFP8, a, b, L.swizzle(sfa), L.swizzle(sfb), M, N, K, out=R.BF16)[1]
    for m in range(M):
        for n in range(N):
            acc = sum(Fraction(ad[m, k]) * Fraction(sa[m, k // 32]) * Fraction(bd[n, k]) * Fraction(sb[n, k // 32])
                      for k in range(K))
            assert abs(Fraction(y[m, n]) - acc) <= abs(acc) * Fraction(1, 2 ** 50)
    assert np.all(np.isfinite(got))


def test_nv_bruteforce_4x4x32_exact():
    M = N = 4
    K = 32
    ac, ap, sfa = _nv_operands(M, K, 3)
    bc, bp, sfb = _nv_operands(N, K, 4)
    sa, sb = _torch_e4m3(sfa), _torch_e4m3(sfb)
    alpha = np.float32(0.375)
    _, y = R.reference(R.NVFP4, ap, bp, L.swizzle(sfa), L.swizzle(sfb), M, N, K, alpha=alpha, out=R.F16)
    for m in range(M):
        for n in range(N):
            acc = sum(Fraction(_e2m1_from_list(ac[m, k])) * Fraction(sa[m, k // 16]) *
                      Fraction(_e2m1_from_list(bc[n, k])) * Fraction(sb[n, k // 16]) for k in range(K))
            assert Fraction(y[m, n]) == Fraction(float(alpha)) * acc       # exact in float64 here


def test_one_hot_rows_select_elements():
    M, N, K = 8, 8, 64
    b, sfb = _mx_operands(N, K, 5)
    a = np.zeros((M, K), dtype=np.uint8)
    sfa = np.full((M, K // 32), 127, dtype=np.uint8)                   # scale 1
    picks = [3, 17, 32, 40, 63, 0, 31, 50]
    for m, k in enumerate(picks):
        a[m, k] = 0x38                                                 # E4M3 1.0
    _, y = R.reference(R.MXFP8, a, b, L.swizzle(sfa), L.swizzle(sfb), M, N, K)
    bd = _torch_e4m3(b) * np.repeat(_torch_e8m0(sfb), 32, axis=1)
    for m, k in enumerate(picks):
        assert np.array_equal(y[m], bd[:, k])


def test_constant_matrices_closed_form():
    M, N, K = 16, 24, 256
    a = np.full((M, K), 0x44, dtype=np.uint8)                          # E4M3 0x44 = 1.5 * 2^1 = 3
    b = np.full((N, K), 0xBA, dtype=np.uint8)                          # -(1.25) = -1.25
    sfa = np.full((M, K // 32), 129, dtype=np.uint8)                   # 4
    sfb = np.full((N, K // 32), 124, dtype=np.uint8)                   # 1/8
    _, y = R.reference(R.MXFP8, a, b, L.swizzle(sfa), L.swizzle(sfb), M, N, K, alpha=2.0)
    assert np.all(y == 2.0 * K * 3.0 * -1.25 * 4 * 0.125)
    # NVFP4: element 0x3 = 1.5, 0xC = -2; scales 0x40 = 2 and 0x30 = 0.5
    ap = np.full((M, K // 2), 0x33, dtype=np.uint8)
    bp = np.full((N, K // 2), 0xCC, dtype=np.uint8)
    _, y2 = R.reference(R.NVFP4, ap, bp, L.swizzle(np.full((M, K // 16), 0x40, np.uint8)),
                        L.swizzle(np.full((N, K // 16), 0x30, np.uint8)), M, N, K)
    assert np.all(y2 == K * 1.5 * -2.0 * 2.0 * 0.5)


def test_operands_are_not_interchangeable():
    M, N, K = 4, 6, 32
    a, sfa = _mx_operands(M, K, 8)
    b, sfb = _mx_operands(N, K, 9)
    _, y = R.reference(R.MXFP8, a, b, L.swizzle(sfa), L.swizzle(sfb), M, N, K)
    ad = _torch_e4m3(a) * np.repeat(_torch_e8m0(sfa), 32, axis=1)
    bd = _torch_e4m3(b) * np.repeat(_torch_e8m0(sfb), 32, axis=1)
    assert y.shape == (M, N)
    for m in range(M):
        for n in range(N):
            assert y[m, n] == pytest.approx(float(np.dot(ad[m], bd[n])), rel=1e-12, abs=1e-300)


def test_naive_loop_matches_library_sum_with_epilogue():
    M, N, K = 5, 7, 64
    xa = synth.normal_rowscaled(M, K, 11)
    xb = synth.normal_rowscaled(N, K, 12)
    ap, sfa, sa = Q.quantize_nvfp4(xa)
    bp, sfb, sb = Q.quantize_nvfp4(xb)
    alpha = np.float32(sa * sb)
    _, bias = synth.bias(N)
    _, y = R.reference(R.NVFP4, ap, bp, L.swizzle(sfa), L.swizzle(sfb), M, N, K, alpha=alpha, bias=bias, silu=True)
    y2 = R.gemm_naive(R.NVFP4, ap, bp, L.swizzle(sfa), L.swizzle(sfb), M, N, K, alpha=alpha, bias=bias, silu=True)
    assert np.allclose(y, y2, rtol=1e-13, atol=1e-15)


def test_epilogue_closed_forms():
    acc = np.array([[0.0, 0.0, 50.0, -50.0]])
    bias = np.array([0.0, 1.0, 0.0, 0.0])
    y = R.epilogue(acc, 1.0, bias, silu=True)
    assert y[0, 0] == 0.0
    assert y[0, 1] == pytest.approx(1.0 / (1.0 + np.exp(-1.0)))
    assert y[0, 2] == pytest.approx(50.0, rel=1e-20)
    assert abs(y[0, 3]) < 1e-19
    # bias goes with the output column
    acc2 = np.zeros((3, 4))
    y2 = R.epilogue(acc2, 1.0, np.arange(4.0), silu=False)
    assert np.array_equal(y2, np.tile(np.arange(4.0), (3, 1)))


def test_tolerance_covers_rounding_only_cases():
    ref = np.array([1.0, 100.0])
    tol = R.tolerance(ref, ref, np.zeros(2), 1.0, False, R.BF16)
    assert np.array_equal(tol, F.ulp_bf16(ref))


def test_residual_and_factor_closed_forms():
    M, N, K = 3, 4, 32
    zero = np.zeros((M, K), dtype=np.uint8)                             # E4M3 0 everywhere: acc = 0
    b, sfb = _mx_operands(N, K, 21)
    sfa = np.full((M, K // 32), 127, dtype=np.uint8)
    C = np.array([[1.5, -2.0, 0.25, 8.0], [0.0, 3.0, -0.5, 1.0], [6.0, -7.0, 0.125, 2.0]])
    bias = np.array([0.25, 0.5, -1.0, 0.0])
    d, y = R.reference(R.MXFP8, zero, b, L.swizzle(sfa), L.swizzle(sfb), M, N, K, bias=bias, C=C, beta=2.0,
                       alpha_row=np.array([3.0, 5.0, 7.0], np.float32), alpha_col=np.ones(N, np.float32))
    assert np.array_equal(y, bias[None, :] + 2.0 * C)                   # small dyadics: exact
    assert np.array_equal(d, y)
    # one-hot rows: D[m, n] = alpha * alpha_row[m] * alpha_col[n] * b_hat[n, k_m]
    a = np.zeros((M, K), dtype=np.uint8)
    picks = [0, 9, 31]
    for m, k in enumerate(picks):
        a[m, k] = 0x38                                                  # 1.0
    ar = np.array([0.5, 2.0, -4.0], dtype=np.float32)
    ac = np.array([1.0, 0.25, -2.0, 8.0], dtype=np.float32)
    _, y2 = R.reference(R.MXFP8, a, b, L.swizzle(sfa), L.swizzle(sfb), M, N, K, alpha=1.5, alpha_row=ar,
                        alpha_col=ac)
    bd = _torch_e4m3(b) * np.repeat(_torch_e8m0(sfb), 32, axis=1)
    for m, k in enumerate(picks):
        for n in range(N):
            assert y2[m, n] == 1.5 * float(ar[m]) * float(ac[n]) * bd[n, k]
    # sampled rows carry their own C row and row factor
    _, y3 = R.reference(R.MXFP8, a, b, L.swizzle(sfa), L.swizzle(sfb), M, N, K, alpha=1.5, alpha_row=ar,
                        alpha_col=ac, C=C, beta=-1.0, rows=[2, 0])
    full = R.reference(R.MXFP8, a, b, L.swizzle(sfa), L.swizzle(sfb), M, N, K, alpha=1.5, alpha_row=ar,
                       alpha_col=ac, C=C, beta=-1.0)[1]
    assert np.array_equal(y3, full[[2, 0]])


def test_naive_loop_matches_with_residual_and_factors():
    M, N, K = 4, 6, 64
    xa = synth.normal_rowscaled(M, K, 13)
    xb = synth.normal_rowscaled(N, K, 14)
    ap, sfa, sa = Q.quantize_nvfp4(xa)
    bp, sfb, sb = Q.quantize_nvfp4(xb)
    rng = np.random.default_rng(15)
    kw = dict(alpha=np.float32(sa * sb), bias=synth.bias(N)[1], silu=True, C=rng.normal(0, 1, (M, N)), beta=0.75,
              alpha_row=rng.uniform(0.5, 2, M).astype(np.float32), alpha_col=rng.uniform(0.5, 2, N).astype(np.float32))
    _, y = R.reference(R.NVFP4, ap, bp, L.swizzle(sfa), L.swizzle(sfb), M, N, K, **kw)
    y2 = R.gemm_naive(R.NVFP4, ap, bp, L.swizzle(sfa), L.swizzle(sfb), M, N, K, **kw)
    assert np.allclose(y, y2, rtol=1e-13, atol=1e-15)


def test_nvfp4_output_closed_form():
    # The NVFP4 output of the epilogue with s = 1 (d = 6): a block whose largest magnitude is 6
    # has scale UE4M3(1) = 0x38 and elements E2M1(y) directly; a block twice as large has scale
    # 0x40 (2) and elements E2M1(y / 2), its 12.000000001 taken as float32 12; a zero block has
    # scale and codes 0; and s = 0 zeroes everything.
    idx = {v: i for i, v in enumerate(E2M1_LIST)}
    vals = [6, 0.5, -1, 1.5, 2, -3, 4, 0.25, 0, 1, -0.5, 3, -6, 2, 1.5, -4]
    # 0.25, the tie between 0 and 0.5, goes to the even code 0
    want = [(idx[abs(v)] | (8 if v < 0 else 0)) if abs(v) != 0.25 else 0 for v in vals]
    y = np.zeros((1, 48))
    y[0, :16] = vals
    y[0, 16:32] = 2 * np.array(vals, dtype=np.float64)
    y[0, 16] = 12.000000001
    codes, scales = R.quantize_output_nvfp4(y, 1.0)
    assert scales.tolist() == [[0x38, 0x40, 0x00]]
    packed = [want[2 * j] | (want[2 * j + 1] << 4) for j in range(8)]
    assert codes[0, :8].tolist() == packed
    assert codes[0, 8:16].tolist() == packed
    assert codes[0, 16:].tolist() == [0] * 8
    codes0, scales0 = R.quantize_output_nvfp4(y, 0.0)
    assert not codes0.any() and not scales0.any()


def test_nvfp4_output_checker_catches_planted_mistakes():
    # The NVFP4-output parity check of the GPU tests, run on the oracle's own output (it must
    # pass, agreeing everywhere) and on that output with a mistake planted: every byte's nibbles
    # swapped, every block scale one code up (both caught by the agreement test), one element
    # code pushed to +-6 where the oracle has 0 (caught by its interval), a nonzero padding
    # byte past M.  Each must fail.
    import parity_util as P
    M, N, K = 130, 48, 64
    prob = P.make_problem("nvfp4", M, N, K, seed_a=7, seed_b=8)
    bias = np.zeros(N)
    _, y = R.reference("nvfp4", prob["A"], prob["B"], prob["SFA"], prob["SFB"], M, N, K, alpha=prob["alpha"],
                       bias=bias, silu=True, out="bf16")
    s = np.float32(np.float32(np.max(np.abs(y))) / np.float32(2688.0))
    codes, scales = R.quantize_output_nvfp4(y, s)
    buf = L.swizzle(scales)
    assert P.check_nvfp4_output(codes.ravel(), buf, prob, bias, True, s) == (1.0, 1.0)
    swapped = ((codes & 0xF) << 4) | (codes >> 4)
    planted = [(swapped.ravel(), buf), (codes.ravel(), L.swizzle(scales + 1))]
    c = codes.copy()
    j = int(np.flatnonzero((c & 0xF) == 0)[0])               # an element (low nibble) coded 0
    c.flat[j] = (c.flat[j] & 0xF0) | 0x7
    planted.append((c.ravel(), buf))
    b2 = buf.copy()
    b2[L.sf_offset(np.array([M + 1]), np.array([0]), N // 16)] = 0x38   # a row past M
    planted.append((codes.ravel(), b2))
    for cd, sb in planted:
        with pytest.raises(AssertionError):
            P.check_nvfp4_output(cd, sb, prob, bias, True, s)


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_parity_tolerance_catches_plausible_mistakes(kind):
    # The element-wise tolerance of the GPU parity tests (|alpha| 2^-7 sum|a b|, x 1.1 with SiLU,
    # + 1 output ulp) must not hide a real mistake: the
    # oracle's own output passes, and that output computed with a mistake planted fails: B's
    # rows in the wrong order, alpha doubled, SiLU left out, the result transposed.  A bias
    # shifted by one column is caught where the accumulation term of the bound vanishes (A all
    # zero: D = round(silu(bias)) up to one output ulp); next to a full accumulation, a bias of
    # N(0, 0.1) sits below 2^-7 sum|a b| and a shift is not visible.
    import parity_util as P
    M, N, K = 64, 64, 256
    prob = P.make_problem(kind, M, N, K, seed_a=21, seed_b=22)
    bias_bits, bias_vals = synth.bias(N, out="bf16")
    silu = True
    ref, _ = P.reference(prob, "bf16", bias_vals, silu)
    P.assert_parity(ref, prob, "bf16", bias_vals, silu)

    def out(p, **kw):
        q = dict(p)
        q.update(kw.pop("prob", {}))
        return P.reference(q, "bf16", kw.get("bias", bias_vals), kw.get("silu", silu))[0]

    perm = np.roll(np.arange(N), 1)
    sfb_lin = L.unswizzle(prob["SFB"], N, K // (32 if kind == "mxfp8" else 16))
    wrong_b = dict(B=prob["B"][perm], SFB=L.swizzle(sfb_lin[perm]))
    planted = [out(prob, prob=wrong_b), out(prob, prob=dict(alpha=np.float32(2 * prob["alpha"]))),
               out(prob, silu=False), ref.T.copy()]
    for got in planted:
        with pytest.raises(AssertionError):
            P.assert_parity(got, prob, "bf16", bias_vals, silu, record=False)
    zero = dict(prob, A=np.zeros_like(prob["A"]))
    zref = out(zero)
    P.assert_parity(zref, zero, "bf16", bias_vals, silu)
    with pytest.raises(AssertionError):
        P.assert_parity(out(zero, bias=np.roll(bias_vals, 1)), zero, "bf16", bias_vals, silu, record=False)


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_secondary_bound_catches_small_mistakes(kind):
    # Mistakes that the stated bar misses, or catches in a few elements only, at K = 4096 must
    # exceed 2^-13 sum|a b| beyond one output ulp, eight times the secondary bound of the GPU
    # parity checks: the oracle's result computed with one block scale of A one code too large
    # (within the stated bar everywhere), and with one k-tile of the kernels (128 E4M3 / 256 E2M1
    # values) left out of every dot product.  The oracle's own result measures 0.
    import parity_util as P
    bound = 2.0 ** -13
    assert P.SECONDARY_REL <= bound / 8
    M, N, K = 128, 128, 4096
    blk = 32 if kind == "mxfp8" else 16
    prob = P.make_problem(kind, M, N, K, seed_a=31, seed_b=32)
    ref, abs_sum = P.reference(prob, "bf16")
    alpha = prob["alpha"]
    assert P.accumulation_ratio(ref, ref, abs_sum, alpha, False, "bf16") == 0.0
    sfa = L.unswizzle(prob["SFA"], M, K // blk).copy()
    sfa[37, 11] += 1
    bumped = P.reference(dict(prob, SFA=L.swizzle(sfa)), "bf16")[0]
    P.assert_parity(bumped, prob, "bf16", record=False)
    assert P.accumulation_ratio(bumped, ref, abs_sum, alpha, False, "bf16") > bound
    # one k-tile dropped: its scales set to code 0 decode to 2^-127 (MXFP8) or 0 (NVFP4)
    kt = 128 if kind == "mxfp8" else 256
    sfa = L.unswizzle(prob["SFA"], M, K // blk).copy()
    sfa[:, 5 * kt // blk:6 * kt // blk] = 0
    dropped = P.reference(dict(prob, SFA=L.swizzle(sfa)), "bf16")[0]
    assert P.accumulation_ratio(dropped, ref, abs_sum, alpha, False, "bf16") > bound
