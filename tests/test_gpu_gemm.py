"""GPU block-scaled GEMM (through the C ABI) against the CPU oracle, element by element.

Bound per output element: |alpha| * 2^-7 * sum_k |a_k b_k| (x 1.1 with SiLU) + 1 output ulp.
Operands are quantised by the oracle; the output buffer carries canaries on both sides.
"""

import os

import numpy as np
import pytest
import torch

import fp4_gemm_blackwell_gb300 as bsg
import parity_util as P
from fp4_gemm_blackwell_gb300 import synth
from oracle import gemm as R

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp8_test_shapes.txt")


def golden_shapes():
    shapes = []
    for line in open(GOLDEN):
        t = line.split()
        if len(t) == 3 and all(s.isdigit() for s in t):
            shapes.append(tuple(int(s) for s in t))
    return shapes


def run_case(kind, M, N, K, out="bf16", bias=False, silu=False, env=None, monkeypatch=None, rows=None):
    if env:
        for k, v in env.items():
            monkeypatch.setenv(k, str(v))
    prob = P.make_problem(kind, M, N, K)
    dp = P.DeviceProblem(prob, out=out, bias=bias, silu=silu)
    with dp.plan() as plan:
        variant = plan.variant
        plan.run()
        plan.check_status()
        got = dp.result()
    P.assert_parity(got, prob, out, dp.bias_vals, silu, rows=rows)
    return variant


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("shape", golden_shapes())
def test_mxfp8_page_shapes(shape, out):
    run_case("mxfp8", *shape, out=out)


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("shape", golden_shapes())
def test_nvfp4_page_shapes_bias_silu(shape, out):
    run_case("nvfp4", *shape, out=out, bias=True, silu=True)


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("M,N,K", [(200, 144, 160), (130, 272, 96), (1, 512, 1024), (16, 4096, 256),
                                   (300, 400, 608)])
def test_ragged_shapes(kind, M, N, K):
    run_case(kind, M, N, K, bias=(kind == "nvfp4"), silu=(kind == "nvfp4"))


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("bn,splits,mode", [(128, 1, ""), (256, 1, ""), (128, 3, "w"), (256, 2, "w"), (128, 7, "w"),
                                            (128, 4, "c"), (128, 8, "c"), (256, 4, "w")])
def test_forced_variants(kind, bn, splits, mode, monkeypatch):
    env = {"BSG_FORCE_BN": bn, "BSG_FORCE_SPLITS": splits}
    if mode == "w":
        env["BSG_SPLIT_WORKSPACE"] = 1
    K = 1792
    v = run_case(kind, 384, 768, K, env=env, monkeypatch=monkeypatch, bias=True, silu=True)
    # a split factor that does not divide the k-tiles evenly is rounded so every split is busy
    # (counted in ring stages: two k-tiles each for 64-wide and unsplit 128-wide tiles)
    kc = 2 if (bn == 64 or (bn == 128 and splits == 1)) and os.environ.get("BSG_KC") != "1" else 1
    if os.environ.get("BSG_KC") == "2" and bn in (64, 128):
        kc = 2
    nkt = -(-K // ((128 if kind == "mxfp8" else 256) * kc))
    kps = -(-nkt // splits)
    s = -(-nkt // kps)
    m = "" if s == 1 else ("w" if mode == "w" or s not in (2, 4, 8) or bn == 256 else "c")
    assert "_bn%d_s%d%s_" % (bn, s, m) in v


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("splits", [2, 4, 8])
def test_cluster_split_64_wide(kind, splits, monkeypatch):
    # 64-wide tiles split over K inside clusters; ragged M and N
    v = run_case(kind, 200, 400, 4096, env={"BSG_FORCE_BN": 64, "BSG_FORCE_SPLITS": splits}, monkeypatch=monkeypatch,
                 bias=True, silu=True)
    assert "_bn64_s%dc_" % splits in v


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_cluster_split_ragged_rows(kind, monkeypatch):
    # ragged M inside a cluster-reduced tile: each CTA's row slab is partly beyond M
    v = run_case(kind, 77, 272, 2048, env={"BSG_FORCE_SPLITS": 4}, monkeypatch=monkeypatch, bias=True, silu=True)
    assert "_s4c_" in v


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("bn", [32, 64])
def test_narrow_tiles(kind, bn, monkeypatch):
    # 32- and 64-wide tiles (B scales taken from a quarter / half of each 128-row band); N = 400
    # leaves the last tile half full, M = 200 a ragged second m-tile
    v = run_case(kind, 200, 400, 1792, env={"BSG_FORCE_BN": bn}, monkeypatch=monkeypatch, bias=True, silu=True)
    assert "_bn%d_s1_" % bn in v


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_narrow_tiles_persistent(kind, monkeypatch):
    # 8 x 128 tiles of 128 x 32 on a persistent grid: every CTA runs several tiles
    v = run_case(kind, 1024, 4096, 512, env={"BSG_FORCE_BN": 32}, monkeypatch=monkeypatch,
                 out="f16", rows=np.arange(0, 1024, 7))
    assert "_bn32_s1_" in v


@pytest.mark.parametrize("M,N,K,expect", [
    (128, 4096, 512, "_bn32_s1_st"),      # short K: 32-wide tiles, no split
    (128, 4096, 4096, "_bn64_s2c_"),      # long K, few tiles: 64-wide tiles, split-K 2 in clusters
    (128, 14336, 1024, "_bn128_s1_"),     # 112 tiles of 128: no split
    (1024, 4096, 1024, "_pair256_"),      # M > 256: CTA pairs
])
def test_default_variants(M, N, K, expect):
    prob = P.make_problem("nvfp4", M, N, K)
    dp = P.DeviceProblem(prob, out="bf16", bias=True, silu=True)
    with dp.plan() as plan:
        assert expect in plan.variant, plan.variant
        plan.run()
        plan.check_status()
        P.assert_parity(dp.result(), prob, "bf16", dp.bias_vals, True, rows=np.arange(0, M, max(1, M // 96)))


def test_narrow_wait_timeout_reports_status(monkeypatch):
    monkeypatch.setenv("BSG_FORCE_BN", "32")
    prob = P.make_problem("nvfp4", 256, 1024, 1024)
    dp = P.DeviceProblem(prob)
    with dp.plan() as plan:
        assert "_bn32_s1_" in plan.variant
        bsg.bsg_plan_debug_set(plan.handle, 1, 50_000_000)
        plan.run()
        with pytest.raises(bsg.BsgError) as e:
            plan.check_status()
        assert e.value.name == "BSG_ERR_DEVICE_TIMEOUT"
        bsg.bsg_plan_debug_set(plan.handle, 0, 0)
        plan.run()
        plan.check_status()
        P.assert_parity(dp.result(), prob, "bf16")


EPI_FAMILIES = [{"BSG_FORCE_PAIR": 1}, {"BSG_FORCE_BN": 256}, {"BSG_FORCE_BN": 128}, {"BSG_FORCE_BN": 64},
                {"BSG_FORCE_BN": 32}, {"BSG_FORCE_BN": 64, "BSG_FORCE_SPLITS": 2},
                {"BSG_FORCE_BN": 128, "BSG_FORCE_SPLITS": 4}, {"BSG_FORCE_BN": 128, "BSG_FORCE_SPLITS": 3}]


@pytest.mark.parametrize("env", EPI_FAMILIES)
@pytest.mark.parametrize("kind,residual,beta,rows_f,cols_f,bias,silu", [
    ("nvfp4", "separate", 0.5, True, True, True, True),      # every term at once
    ("mxfp8", "inplace", -1.0, False, True, False, False),   # D += A B^T scaled per column, in place
    ("nvfp4", None, 0.0, True, False, True, False),          # per-row factor alone
])
def test_residual_and_factor_epilogue(env, kind, residual, beta, rows_f, cols_f, bias, silu, monkeypatch):
    # beta * C and alpha * alpha_row[m] * alpha_col[n] through every epilogue path: one and two
    # TMEM accumulators, CTA pairs, split-K reduced in a cluster and through the workspace
    for k, v in env.items():
        monkeypatch.setenv(k, str(v))
    prob = P.make_problem(kind, 300, 272, 2048)   # K: 2, 3 and 4 splits stay exact for both formats
    dp = P.DeviceProblem(prob, out="bf16", bias=bias, silu=silu, residual=residual, beta=beta,
                         alpha_row=rows_f, alpha_col=cols_f)
    with dp.plan() as plan:
        variant = plan.variant
        plan.run()
        plan.check_status()
        got = dp.result()
    if "BSG_FORCE_SPLITS" in env:
        assert ("_s%d" % env["BSG_FORCE_SPLITS"]) in variant, variant
    P.assert_parity(got, prob, "bf16", dp.bias_vals, silu, epi=dp.epi_kwargs())


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("env", [{"BSG_FORCE_PAIR": 1}, {"BSG_FORCE_BN": 256}, {"BSG_FORCE_BN": 128},
                                 {"BSG_FORCE_BN": 64}, {"BSG_FORCE_BN": 32}])
def test_output_only_16_byte_aligned(kind, env, monkeypatch):
    # D 16 bytes past a 32-byte boundary: the epilogues fall back from 32-byte to 16-byte stores
    for k, v in env.items():
        monkeypatch.setenv(k, str(v))
    prob = P.make_problem(kind, 300, 272, 512)
    dp = P.DeviceProblem(prob, out="bf16", bias=True, silu=kind == "nvfp4", margin=8)
    assert dp.D.data_ptr() % 32 == 16
    with dp.plan() as plan:
        plan.run()
        plan.check_status()
        got = dp.result()
    P.assert_parity(got, prob, "bf16", dp.bias_vals, kind == "nvfp4")


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("M,N,K,out", [(256, 256, 512, "bf16"), (300, 272, 1024, "f16"), (2048, 2560, 512, "bf16"),
                                       (640, 768, 4096, "bf16"),
                                       # K past the last whole stage (NVFP4 stages take 256 of K,
                                       # MXFP8 128): a last stage of 1 or 3 MMAs, its scale boxes
                                       # reaching past K
                                       (512, 512, 1056, "bf16"), (320, 512, 1184, "bf16")])
def test_pair_kernel(kind, M, N, K, out, monkeypatch):
    # CTA-pair kernel (256 x 256 tiles on 2-CTA clusters): ragged M and N, both outputs,
    # more pair tiles than SM pairs (persistent loop)
    v = run_case(kind, M, N, K, out=out, env={"BSG_FORCE_PAIR": 1}, monkeypatch=monkeypatch,
                 bias=(kind == "nvfp4"), silu=(kind == "nvfp4"))
    assert "_pair256_" in v


def test_pair_wait_timeout_reports_status(monkeypatch):
    monkeypatch.setenv("BSG_FORCE_PAIR", "1")
    prob = P.make_problem("nvfp4", 512, 512, 1024)
    dp = P.DeviceProblem(prob)
    with dp.plan() as plan:
        assert "_pair256_" in plan.variant
        bsg.bsg_plan_debug_set(plan.handle, 1, 50_000_000)
        plan.run()
        with pytest.raises(bsg.BsgError) as e:
            plan.check_status()
        assert e.value.name == "BSG_ERR_DEVICE_TIMEOUT"
        bsg.bsg_plan_debug_set(plan.handle, 0, 0)
        plan.run()
        plan.check_status()
        P.assert_parity(dp.result(), prob, "bf16")


def test_pdl_off_matches(monkeypatch):
    run_case("nvfp4", 256, 512, 1024, env={"BSG_PDL": 0}, monkeypatch=monkeypatch, bias=True, silu=True)


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_persistent_multi_tile_per_cta(kind, monkeypatch):
    # 16 x 10 = 160 tiles of 128 x 256 on 152 SMs: some CTAs run two tiles (1-SM kernel)
    v = run_case(kind, 2048, 2560, 512, env={"BSG_FORCE_PAIR": 0}, monkeypatch=monkeypatch)
    assert "_bn256_s1_" in v


def test_device_alpha_and_repeat_runs():
    prob = P.make_problem("nvfp4", 256, 512, 512)
    dp = P.DeviceProblem(prob, out="bf16", bias=True, silu=True)
    alpha = torch.tensor([float(prob["alpha"])], dtype=torch.float32, device="cuda")
    with dp.plan(alpha_dev=alpha) as plan:
        for _ in range(3):
            plan.run()
        plan.check_status()
        P.assert_parity(dp.result(), prob, "bf16", dp.bias_vals, True)


def test_one_shot_calls_match_oracle():
    bsg.bsg_cache_clear()
    for kind in ("mxfp8", "nvfp4"):
        prob = P.make_problem(kind, 192, 256, 384)
        dp = P.DeviceProblem(prob, out="bf16", bias=(kind == "nvfp4"), silu=(kind == "nvfp4"))
        for _ in range(2):                       # second call is a plan-cache hit
            if kind == "mxfp8":
                bsg.mxfp8_gemm(dp.D, dp.A, dp.B, dp.SFA, dp.SFB, float(prob["alpha"]), 192, 256, 384,
                               bsg.BSG_OUT_BF16)
            else:
                bsg.nvfp4_gemm(dp.D, dp.A, dp.B, dp.SFA, dp.SFB, dp.bias, float(prob["alpha"]), dp.flags,
                               192, 256, 384, bsg.BSG_OUT_BF16)
            P.assert_parity(dp.result(), prob, "bf16", dp.bias_vals, kind == "nvfp4")
    bsg.bsg_cache_clear()


def test_undersized_scale_buffer_is_rejected():
    prob = P.make_problem("mxfp8", 256, 256, 256)
    dp = P.DeviceProblem(prob)
    # the caching allocator sub-allocates large segments: take the last 512 bytes of a fresh
    # 64 MiB segment, so that the 2048-byte scale buffer would run past the allocation's end
    torch.cuda.empty_cache()
    seg = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    tail = seg[(64 << 20) - 512:]
    with pytest.raises(bsg.BsgError) as e:
        bsg.bsg_plan_create(bsg.BSG_MXFP8, bsg.BSG_OUT_BF16, 256, 256, 256, dp.A, dp.B, tail, dp.SFB, dp.D)
    assert e.value.name == "BSG_ERR_SCALE_LAYOUT"


def test_wait_timeout_reports_status_and_context_survives():
    prob = P.make_problem("mxfp8", 256, 256, 256)
    dp = P.DeviceProblem(prob)
    with dp.plan() as plan:
        bsg.bsg_plan_debug_set(plan.handle, 1, 50_000_000)       # 50 ms limit, first stage never loaded
        plan.run()
        with pytest.raises(bsg.BsgError) as e:
            plan.check_status()
        assert e.value.name == "BSG_ERR_DEVICE_TIMEOUT"
        bsg.bsg_plan_debug_set(plan.handle, 0, 0)
        plan.run()
        plan.check_status()
        P.assert_parity(dp.result(), prob, "bf16")



def _batched_buffers(kind, L, M, N, K, pad=256, residual=False):
    """L problems quantised by the oracle, copied into single device buffers at strides of one
    entry + pad bytes; D with canaries between the entries."""
    probs = [P.make_problem(kind, M, N, K, seed_a=10 + l, seed_b=20 + l) for l in range(L)]
    def pack(arrs):
        one = max(a.size for a in arrs)
        stride = (one + pad + 15) // 16 * 16
        buf = np.full(L * stride, 0x5A, dtype=np.uint8)
        for l, a in enumerate(arrs):
            buf[l * stride:l * stride + a.size] = np.ascontiguousarray(a).view(np.uint8).ravel()
        return P.dev(buf), stride
    A, sA = pack([p["A"] for p in probs])
    B, sB = pack([p["B"] for p in probs])
    SFA, sSFA = pack([p["SFA"] for p in probs])
    SFB, sSFB = pack([p["SFB"] for p in probs])
    sD = (M * N * 2 + pad + 15) // 16 * 16
    D = torch.full((L * sD // 2,), 0x7BAD, dtype=torch.int16, device="cuda")
    C = Cvals = None
    sC = 0
    if residual:
        sC = sD
        bits = np.zeros(L * sC // 2, dtype=np.uint16)
        Cvals = []
        for l in range(L):
            b, v = P.synth_residual(M, N, "bf16", seed=40 + l)
            bits[l * sC // 2:l * sC // 2 + M * N] = b.ravel()
            Cvals.append(v)
        C = P.dev(bits.view(np.int16)).view(torch.int16)
    strides = dict(stride_A=sA, stride_B=sB, stride_SFA=sSFA, stride_SFB=sSFB, stride_D=sD, stride_C=sC)
    return probs, A, B, SFA, SFB, D, C, Cvals, strides


@pytest.mark.parametrize("env", [{}, {"BSG_FORCE_PAIR": 1}, {"BSG_FORCE_BN": 256}, {"BSG_FORCE_BN": 128},
                                 {"BSG_FORCE_BN": 32}, {"BSG_FORCE_BN": 64, "BSG_FORCE_SPLITS": 2},
                                 {"BSG_FORCE_BN": 128, "BSG_FORCE_SPLITS": 3}])
@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_batched(kind, env, monkeypatch):
    # L = 3 problems of one shape in one launch (the L of the {m, n, k, l} problem shape), every
    # kernel family; each entry against its own oracle result, nothing written between entries
    for k, v in env.items():
        monkeypatch.setenv(k, str(v))
    L, M, N, K = 3, 200, 144, 1536
    residual = kind == "nvfp4" and "BSG_FORCE_SPLITS" in env
    probs, A, B, SFA, SFB, D, C, Cvals, strides = _batched_buffers(kind, L, M, N, K, residual=residual)
    bias_bits, bias_vals = synth.bias(N, out="bf16")
    bias = P.dev(bias_bits.view(np.int16)).view(torch.int16)
    flags = bsg.BSG_F_BIAS | (bsg.BSG_F_SILU if kind == "nvfp4" else 0) | (bsg.BSG_F_C if residual else 0)
    alphas = [float(p["alpha"]) for p in probs]
    # alpha is shared by the batch: give every entry the same one by scaling with entry 0's
    alpha = alphas[0]
    D2 = torch.full_like(D, 0x7BAD)
    with bsg.Plan(P.KIND[kind], P.OUT["bf16"], M, N, K, A, B, SFA, SFB, D, alpha=alpha, flags=flags, bias=bias,
                  C=C, beta=0.5, L=L, strides=strides) as plan:
        variant = plan.variant
        plan.run()
        plan.run_operands(A, B, SFA, SFB, D2, bias=bias, C=C)  # 3-D maps rewritten on the device
        plan.check_status()
    torch.cuda.synchronize()
    dall = D.cpu().numpy().view(np.uint16)
    assert np.array_equal(D2.cpu().numpy().view(np.uint16), dall), variant
    sD = strides["stride_D"] // 2
    for l, p in enumerate(probs):
        got = R.out_from_bits(dall[l * sD:l * sD + M * N].reshape(M, N), "bf16")
        q = dict(p)
        q["alpha"] = np.float32(alpha)
        epi = dict(C=Cvals[l], beta=0.5) if residual else None
        P.assert_parity(got, q, "bf16", bias_vals, kind == "nvfp4", epi=epi)
        gap = dall[l * sD + M * N:(l + 1) * sD] if l + 1 < L else dall[l * sD + M * N:]
        assert np.all(gap == 0x7BAD), "wrote past entry %d (%s)" % (l, variant)


def _grouped_layout(sizes, tail):
    """Rows of groups of the given sizes, each starting on a multiple of 128 and padded with -1
    rows to the next one, then `tail` rows of no group.  Returns (group_index, rows of each group)."""
    idx, rows, at = [], [], 0
    for g, n in enumerate(sizes):
        pad = -n % 128
        rows.append(list(range(at, at + n)))
        idx += [g] * n + [-1] * pad
        at += n + pad
    idx += [-1] * tail
    return np.array(idx, dtype=np.int32), rows


@pytest.mark.parametrize("env", [{}, {"BSG_FORCE_BN": 256}, {"BSG_FORCE_BN": 128}, {"BSG_FORCE_BN": 32},
                                 {"BSG_FORCE_BN": 64, "BSG_FORCE_SPLITS": 2},
                                 {"BSG_FORCE_BN": 128, "BSG_FORCE_SPLITS": 3},
                                 {"BSG_FORCE_PAIR": 1}])
@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_grouped(kind, env, monkeypatch):
    # Grouped GEMM (expert GEMMs of a mixture-of-experts layer): 4 groups of 200, 0, 37 and 128
    # rows with their own B and alpha, in the 128-row-aligned layout; then a block whose first
    # row names group 99 (skipped whole) and a ragged tail of no group.  One row inside group
    # 3's block is marked group 2: it is not stored.  Each group against its own oracle result;
    # every row of no stored group keeps the canary.  A forced CTA pair must not apply to a
    # grouped problem.
    for k, v in env.items():
        monkeypatch.setenv(k, str(v))
    G, N, K = 4, 144, 1536
    gidx, grows = _grouped_layout([200, 0, 37, 128], tail=0)
    stray = grows[3][5]
    gidx[stray] = 2
    grows[3].remove(stray)
    skip_block = np.zeros(128, dtype=np.int32)
    skip_block[0] = 99
    gidx = np.concatenate([gidx, skip_block, np.full(60, -1, dtype=np.int32)])
    M = len(gidx)
    gen = synth.normal_rowscaled if kind == "nvfp4" else synth.normal
    a, sfa, sa = P.oracle_operand(kind, gen(M, K, 31))
    bs = [P.oracle_operand(kind, gen(N, K, 40 + g)) for g in range(G)]
    if kind == "nvfp4":
        alphas = [np.float32(np.float32(sa) * np.float32(s)) for _, _, s in bs]
    else:
        alphas = [np.float32(x) for x in (1.0, 0.5, 2.0, 0.25)]

    def pack(arrs, pad=256):
        one = max(x.size for x in arrs)
        stride = (one + pad + 15) // 16 * 16
        buf = np.full(G * stride, 0x5A, dtype=np.uint8)
        for g, x in enumerate(arrs):
            buf[g * stride:g * stride + x.size] = np.ascontiguousarray(x).view(np.uint8).ravel()
        return P.dev(buf), stride

    B, sB = pack([b for b, _, _ in bs])
    SFB, sSFB = pack([f for _, f, _ in bs])
    A, SFA = P.dev(a), P.dev(sfa)
    alpha_dev = torch.tensor(np.array(alphas, dtype=np.float32), device="cuda")
    gi = torch.from_numpy(gidx).cuda()
    D = torch.full((M * N,), 0x7BAD, dtype=torch.int16, device="cuda")
    residual = "BSG_FORCE_SPLITS" in env
    C = Cvals = None
    if residual:
        cbits, Cvals = P.synth_residual(M, N, "bf16", seed=77)
        C = P.dev(cbits.view(np.int16)).view(torch.int16)
    bias_bits, bias_vals = synth.bias(N, out="bf16")
    bias = P.dev(bias_bits.view(np.int16)).view(torch.int16)
    silu = kind == "nvfp4"
    flags = (bsg.BSG_F_GROUPED | bsg.BSG_F_ALPHA_DEVICE | bsg.BSG_F_BIAS | (bsg.BSG_F_SILU if silu else 0) |
             (bsg.BSG_F_C if residual else 0))
    D2 = torch.full_like(D, 0x7BAD)
    with bsg.Plan(P.KIND[kind], P.OUT["bf16"], M, N, K, A, B, SFA, SFB, D, flags=flags, bias=bias,
                  alpha_dev=alpha_dev, C=C, beta=0.75, L=G, strides=dict(stride_B=sB, stride_SFB=sSFB),
                  group_index=gi) as plan:
        variant = plan.variant
        plan.run()
        plan.run_operands(A, B, SFA, SFB, D2, bias=bias, alpha_dev=alpha_dev, C=C, group_index=gi)
        plan.check_status()
    torch.cuda.synchronize()
    assert np.array_equal(D2.cpu().numpy(), D.cpu().numpy()), variant
    assert "pair" not in variant, variant
    bits = D.cpu().numpy().view(np.uint16).reshape(M, N)
    got = R.out_from_bits(bits, "bf16")
    stored = np.zeros(M, dtype=bool)
    for g in range(G):
        if not grows[g]:
            continue
        b, sfb, _ = bs[g]
        prob = dict(kind=kind, M=M, N=N, K=K, A=a, B=b, SFA=sfa, SFB=sfb, alpha=alphas[g])
        epi = dict(C=Cvals, beta=0.75) if residual else None
        P.assert_parity(got, prob, "bf16", bias_vals, silu, rows=grows[g], epi=epi)
        stored[grows[g]] = True
    assert np.all(bits[~stored] == 0x7BAD), "rows of no stored group were written (%s)" % variant


@pytest.mark.parametrize("env", [{}, {"BSG_FORCE_PAIR": 1}, {"BSG_FORCE_BN": 256}, {"BSG_FORCE_BN": 32},
                                 {"BSG_FORCE_BN": 64, "BSG_FORCE_SPLITS": 2},
                                 {"BSG_FORCE_BN": 128, "BSG_FORCE_SPLITS": 3}])
@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_run_operands(kind, env, monkeypatch):
    # Pointer-agnostic runs: one plan, made on problem 1's buffers, runs on problem 2's (its
    # tensor maps rewritten on the device), then plainly on its own, then on problem 2's again;
    # every kernel family (CTA pair, one and two accumulators, split-K in a cluster and through
    # the workspace).  Each result against its own oracle; the other D untouched.
    for k, v in env.items():
        monkeypatch.setenv(k, str(v))
    silu = kind == "nvfp4"
    p1 = P.make_problem(kind, 300, 272, 2048, seed_a=3, seed_b=4)
    p2 = P.make_problem(kind, 300, 272, 2048, seed_a=5, seed_b=6)
    d1 = P.DeviceProblem(p1, bias=True, silu=silu, residual="separate", beta=0.5)
    d2 = P.DeviceProblem(p2, bias=True, silu=silu, residual="separate", beta=0.5)
    a1 = torch.tensor([float(p1["alpha"])], dtype=torch.float32, device="cuda")
    a2 = torch.tensor([float(p2["alpha"])], dtype=torch.float32, device="cuda")

    def run2(plan):
        plan.run_operands(d2.A, d2.B, d2.SFA, d2.SFB, d2.D, bias=d2.bias, alpha_dev=a2, C=d2.C)

    with d1.plan(alpha_dev=a1) as plan:
        variant = plan.variant
        run2(plan)
        plan.check_status()
        got2 = d2.result()
        assert np.all(d1.Dbuf.cpu().numpy().view(np.uint16) == d1.CANARY), "the plan's own D was written"
        plan.run()
        plan.check_status()
        got1 = d1.result()
        d2.Dbuf.fill_(d2.CANARY)
        run2(plan)
        plan.check_status()
        got2b = d2.result()
    P.assert_parity(got2, p2, "bf16", d2.bias_vals, silu, epi=d2.epi_kwargs())
    P.assert_parity(got1, p1, "bf16", d1.bias_vals, silu, epi=d1.epi_kwargs())
    assert np.array_equal(got2, got2b), variant
    if "BSG_FORCE_PAIR" in env:
        assert "pair" in variant, variant


def _nvfp4_output_case(kind, env, M, N, K, extra, monkeypatch):
    """One GEMM with NVFP4 output under `env`, checked against the oracle (see test_nvfp4_output);
    returns the plan's variant."""
    for k, v in env.items():
        monkeypatch.setenv(k, str(v))
    silu = kind == "nvfp4"
    prob = P.make_problem(kind, M, N, K, seed_a=7, seed_b=8)
    bias_bits, bias_vals = synth.bias(N, out="bf16")
    bias = P.dev(bias_bits.view(np.int16)).view(torch.int16)
    epi, C, ar, ac = None, None, None, None
    if extra:
        cbits, cvals = P.synth_residual(M, N, "bf16", seed=11)
        rng = np.random.default_rng(12)
        arv = rng.uniform(0.5, 2.0, M).astype(np.float32)
        acv = rng.uniform(0.5, 2.0, N).astype(np.float32)
        C = P.dev(cbits.view(np.int16)).view(torch.int16)
        ar, ac = P.dev(arv).view(torch.float32), P.dev(acv).view(torch.float32)
        epi = dict(C=cvals, beta=0.5, alpha_row=arv, alpha_col=acv)
    _, y = R.reference(kind, prob["A"], prob["B"], prob["SFA"], prob["SFB"], M, N, K, alpha=prob["alpha"],
                       bias=bias_vals, silu=silu, out="bf16", **(epi or {}))
    s = np.float32(np.float32(np.max(np.abs(y))) / np.float32(2688.0))   # the recipe's tensor scale
    d_scale = torch.tensor([float(s)], dtype=torch.float32, device="cuda")
    nsf = bsg.bsg_sf_bytes(bsg.BSG_NVFP4, M, N)
    pad = 256

    def buffers():
        dbuf = torch.full((M * N // 2 + 2 * pad,), 0xCD, dtype=torch.uint8, device="cuda")
        sbuf = torch.full((nsf + 2 * pad,), 0xAB, dtype=torch.uint8, device="cuda")
        return dbuf, sbuf, dbuf[pad:pad + M * N // 2], sbuf[pad:pad + nsf]

    dbuf, sbuf, D, SFD = buffers()
    dbuf2, sbuf2, D2, SFD2 = buffers()
    A, B, SFA, SFB = P.dev(prob["A"]), P.dev(prob["B"]), P.dev(prob["SFA"]), P.dev(prob["SFB"])
    flags = bsg.BSG_F_BIAS | (bsg.BSG_F_SILU if silu else 0)
    if extra:
        flags |= bsg.BSG_F_C | bsg.BSG_F_ALPHA_ROW | bsg.BSG_F_ALPHA_COL
    with bsg.Plan(P.KIND[kind], bsg.BSG_OUT_NVFP4, M, N, K, A, B, SFA, SFB, D, alpha=float(prob["alpha"]),
                  flags=flags, bias=bias, C=C, beta=0.5, alpha_row=ar, alpha_col=ac, SFD=SFD, d_scale=d_scale) as plan:
        variant = plan.variant
        plan.run()
        plan.run_operands(A, B, SFA, SFB, D2, bias=bias, C=C, alpha_row=ar, alpha_col=ac, SFD=SFD2, d_scale=d_scale)
        plan.check_status()
    torch.cuda.synchronize()
    db, sb = dbuf.cpu().numpy(), sbuf.cpu().numpy()
    assert np.all(db[:pad] == 0xCD) and np.all(db[-pad:] == 0xCD), "D margins written (%s)" % variant
    assert np.all(sb[:pad] == 0xAB) and np.all(sb[-pad:] == 0xAB), "SFD margins written (%s)" % variant
    P.check_nvfp4_output(db[pad:-pad], sb[pad:-pad], prob, bias_vals, silu, s, epi=epi)
    assert np.array_equal(dbuf2.cpu().numpy(), db) and np.array_equal(sbuf2.cpu().numpy(), sb), variant
    return variant


@pytest.mark.parametrize("env", [{}, {"BSG_FORCE_BN": 64}, {"BSG_FORCE_BN": 128}, {"BSG_FORCE_BN": 256},
                                 {"BSG_FORCE_PAIR": 1}, {"BSG_FORCE_BN": 32}, {"BSG_FORCE_BN": 128, "BSG_FORCE_SPLITS": 2}])
@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_nvfp4_output(kind, env, monkeypatch):
    # D written as NVFP4 (E2M1 codes + swizzled UE4M3 scales, global scale from the device) by
    # every unsplit kernel family (and the default choice); M and N ragged (N/16 = 17 scale columns: 3 of padding), bias
    # (+ SiLU), and with some families the residual and both factor vectors.  Checked by intervals
    # and agreement against the oracle's quantisation of its own result, the scale padding zero,
    # the buffers' margins untouched; a split forced on 128-wide tiles does not apply (the
    # split-K reductions encode NVFP4 on 64-wide tiles); a pointer-agnostic run into second
    # buffers gives the same bytes.
    variant = _nvfp4_output_case(kind, env, 300, 272, 1024, env.get("BSG_FORCE_BN") in (64, 256), monkeypatch)
    if env:
        assert "_s1" in variant or "pair" in variant, variant


@pytest.mark.parametrize("env,extra", [
    ({"BSG_FORCE_BN": 64, "BSG_FORCE_SPLITS": 2}, False),      # cluster reduction, 2 splits
    ({"BSG_FORCE_BN": 64, "BSG_FORCE_SPLITS": 4}, True),       # cluster reduction, 4, residual + factors
    ({"BSG_FORCE_BN": 64, "BSG_FORCE_SPLITS": 3}, True),       # through the workspace (3 splits)
    ({"BSG_FORCE_BN": 64, "BSG_FORCE_SPLITS": 2, "BSG_SPLIT_WORKSPACE": 1}, False),
])
@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_nvfp4_output_split_k(kind, env, extra, monkeypatch):
    # NVFP4 output from the split-K reductions: in a cluster each block of 16 columns is encoded
    # by four lanes that share its amax, through the workspace by the last split's row segments.
    # M = 300 leaves rows of the last tile without a problem row (their scales zero), N = 272 puts
    # scale columns 17..19 (padding) in the last 64-wide tile.
    variant = _nvfp4_output_case(kind, env, 300, 272, 4096, extra, monkeypatch)
    want = "_s%d%s_" % (env["BSG_FORCE_SPLITS"],
                        "w" if ("BSG_SPLIT_WORKSPACE" in env or env["BSG_FORCE_SPLITS"] == 3) else "c")
    assert "_bn64" in variant and want in variant, variant


def test_nvfp4_output_skinny_default_splits(monkeypatch):
    # the skinny shape with NVFP4 output takes the split-K variant of its 16-bit-output twin
    variant = _nvfp4_output_case("nvfp4", {}, 128, 4096, 4096, False, monkeypatch)
    assert "_bn64_s2c_" in variant, variant


@pytest.mark.parametrize("env", [{}, {"BSG_FORCE_BN": 64, "BSG_FORCE_SPLITS": 2}, {"BSG_FORCE_PAIR": 1}])
def test_batched_device_alpha_per_entry(env, monkeypatch):
    # L = 3 NVFP4 problems whose global factors differ (each entry's s_A * s_B): with
    # BSG_F_ALPHA_DEVICE, alpha_dev holds one alpha per entry, and each entry matches its own
    # oracle result with its own alpha
    for k, v in env.items():
        monkeypatch.setenv(k, str(v))
    L, M, N, K = 3, 300, 144, 1024
    probs, A, B, SFA, SFB, D, _, _, strides = _batched_buffers("nvfp4", L, M, N, K)
    alphas = np.array([p["alpha"] for p in probs], dtype=np.float32)
    assert len(set(alphas.tolist())) == L
    ad = torch.from_numpy(alphas).cuda()
    with bsg.Plan(bsg.BSG_NVFP4, bsg.BSG_OUT_BF16, M, N, K, A, B, SFA, SFB, D, flags=bsg.BSG_F_ALPHA_DEVICE,
                  alpha_dev=ad, L=L, strides=strides) as plan:
        variant = plan.variant
        plan.run()
        plan.check_status()
    torch.cuda.synchronize()
    dall = D.cpu().numpy().view(np.uint16)
    sD = strides["stride_D"] // 2
    for l, p in enumerate(probs):
        got = R.out_from_bits(dall[l * sD:l * sD + M * N].reshape(M, N), "bf16")
        P.assert_parity(got, p, "bf16")
    if "BSG_FORCE_PAIR" in env:
        assert "pair" in variant, variant


@pytest.mark.parametrize("env", EPI_FAMILIES)
@pytest.mark.parametrize("kind,residual", [("nvfp4", None), ("mxfp8", None), ("nvfp4", "separate"),
                                           ("mxfp8", "inplace")])
def test_additive_terms_where_rows_of_a_are_zero(env, kind, residual, monkeypatch):
    # Rows of A that are all zero have an accumulation term of exactly 0, so there the output is
    # the epilogue's additive terms alone: D[m, n] = round(silu(bias[n] + beta * C[m, n])) to one
    # output ulp, a bound too tight for a bias or C taken from a neighbouring column or row.  The
    # zero rows are scattered over lanes, warps and tiles; the other rows check the accumulation
    # in the same launch.  Every kernel family, the plain instantiation (bias + SiLU) and the
    # extended one (with C).
    for k, v in env.items():
        monkeypatch.setenv(k, str(v))
    M, N, K = 300, 272, 2048
    zero = (np.arange(M) // 7) % 3 == 0
    prob = P.make_problem(kind, M, N, K, zero_rows=zero)
    assert not prob["A"][zero].any()
    dp = P.DeviceProblem(prob, out="bf16", bias=True, silu=True, residual=residual, beta=0.75)
    with dp.plan() as plan:
        variant = plan.variant
        plan.run()
        plan.check_status()
        got = dp.result()
    P.assert_parity(got, prob, "bf16", dp.bias_vals, True, epi=dp.epi_kwargs())
    # the closed form of the zero rows, written out here rather than taken from the oracle
    y = np.broadcast_to(dp.bias_vals[None, :], (M, N)).astype(np.float64)
    if residual is not None:
        y = y + np.float64(np.float32(0.75)) * dp.C_vals
    y = y / (1.0 + np.exp(-y))
    want = R.round_out(y, "bf16")[zero]
    g = got[zero]
    ulp = R.ulp_out(np.maximum(np.abs(want), np.abs(g)), "bf16")
    bad = np.abs(g - want) > ulp
    assert not bad.any(), "%s: %d zero-row outputs off by more than one ulp, first at %s" % (
        variant, bad.sum(), np.argwhere(bad)[:3].tolist())
