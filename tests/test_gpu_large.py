"""GPU parity at the pages' full-size configurations, against the CPU oracle on sampled rows.

The configurations of the block-scaled GEMM pages that the benchmark times:
  * MXFP8 8192 x 8192 x 8192 with FP16 and with BF16 output;
  * NVFP4 8192 x 8192 x 8192 with BF16 bias and SiLU, BF16 output, and the ragged
    M = 8000 variant (M not a multiple of the tile);
  * the shapes of the launch-overhead loop: NVFP4 M in {1, 16, 128, 1024} x (N, K) in
    {(4096, 4096), (14336, 4096), (4096, 14336)}, BF16 output, through the one-shot call.
Every operand is quantised by the oracle (row chunks in spawned worker processes) and uploaded;
each run goes through the plan (or the one-shot call) that the benchmark uses, so the kernel
variant under test is the timed one.  The oracle's float64 result is computed for sampled rows
(every 61st row, which visits every lane position of the 128-row tiles, plus the last rows of a
ragged M) over all N columns, and compared element by element with the parity bound of the
other GEMM tests.  The output buffers carry canaries on both sides.
"""

import numpy as np
import pytest
import torch

import fp4_gemm_blackwell_gb300 as bsg
import oracle_pool
import parity_util as P
from fp4_gemm_blackwell_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

_OPERANDS = {}


@pytest.fixture(scope="module")
def pool():
    p = oracle_pool.spawn_pool()
    yield p
    p.close()
    p.join()


def operand(pool, kind, rows, K, seed):
    """The oracle's (codes, swizzled scales, s) of the seeded rows x K operand (cached per module)."""
    key = (kind, rows, K, seed)
    if key not in _OPERANDS:
        gen = synth.normal_rowscaled if kind == "nvfp4" else synth.normal
        _OPERANDS[key] = oracle_pool.operand(kind, gen(rows, K, seed), pool)
    return _OPERANDS[key]


def problem(pool, kind, M, N, K):
    a, sfa, sa = operand(pool, kind, M, K, synth.SEED_A)
    b, sfb, sb = operand(pool, kind, N, K, synth.SEED_B)
    alpha = np.float32(1.0) if kind == "mxfp8" else np.float32(np.float32(sa) * np.float32(sb))
    return dict(kind=kind, M=M, N=N, K=K, A=a, B=b, SFA=sfa, SFB=sfb, alpha=alpha)


def sample_rows(M, tail=0):
    rows = set(range(0, M, 61)) | set(range(max(0, M - tail), M)) | {M - 1}
    return np.array(sorted(rows))


@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_mxfp8_8192_cube(pool, out):
    prob = problem(pool, "mxfp8", 8192, 8192, 8192)
    dp = P.DeviceProblem(prob, out=out)
    with dp.plan() as plan:
        assert "_pair256_" in plan.variant, plan.variant
        plan.run()
        plan.check_status()
        got = dp.result()
    P.assert_parity(got, prob, out, rows=sample_rows(8192))


@pytest.mark.parametrize("M", [8192, 8000])
def test_nvfp4_8192_cube_bias_silu(pool, M):
    prob = problem(pool, "nvfp4", M, 8192, 8192)
    dp = P.DeviceProblem(prob, out="bf16", bias=True, silu=True)
    with dp.plan() as plan:
        assert "_pair256_" in plan.variant, plan.variant
        plan.run()
        plan.check_status()
        got = dp.result()
    P.assert_parity(got, prob, "bf16", dp.bias_vals, True, rows=sample_rows(M, tail=64))


@pytest.mark.parametrize("N,K", [(4096, 4096), (14336, 4096), (4096, 14336)])
@pytest.mark.parametrize("M", [1, 16, 128, 1024])
def test_launch_loop_shapes(pool, M, N, K):
    prob = problem(pool, "nvfp4", M, N, K)
    dp = P.DeviceProblem(prob, out="bf16")
    bsg.bsg_cache_clear()
    for _ in range(2):                      # a plan-cache miss, then a hit
        dp.Dbuf.fill_(dp.CANARY)
        bsg.nvfp4_gemm(dp.D, dp.A, dp.B, dp.SFA, dp.SFB, None, float(prob["alpha"]), 0, M, N, K,
                       bsg.BSG_OUT_BF16)
        got = dp.result()
        rows = np.arange(M) if M <= 128 else sample_rows(M)
        P.assert_parity(got, prob, "bf16", rows=rows)
    bsg.bsg_cache_clear()
    torch.cuda.synchronize()
