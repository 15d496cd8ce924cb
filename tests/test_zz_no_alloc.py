"""The allocation-free GEMM entry point against the plan entry point.

bsg_gemm_noalloc is for callers that may not allocate device memory when they run a GEMM
(allocator callbacks, engines with a fixed device-memory budget); it keeps its scratch in a
static device array instead of a plan's workspace.  Here it is called through the C ABI twice
in a row per problem and each output is compared with bsg_plan_run's output on the same
operands, within the parity tolerance the other GEMM tests use.  This file is collected last.
"""

import numpy as np
import pytest
import torch

import fp4_gemm_blackwell_gb300 as bsg
import parity_util as P
from oracle import gemm as R

pytestmark = pytest.mark.gpu


def _call_noalloc(dp, prob):
    p = prob
    dp.Dbuf.fill_(dp.CANARY)
    bsg.bsg_gemm_noalloc(P.KIND[p["kind"]], P.OUT[dp.out], p["M"], p["N"], p["K"], dp.A, dp.B, dp.SFA, dp.SFB,
                         dp.D, alpha=float(p["alpha"]), flags=dp.flags, bias=dp.bias)
    return dp.result()


@pytest.mark.parametrize("kind,M,N,K,epi,workspace", [
    ("nvfp4", 128, 512, 4096, True, True),    # split-K through scratch: partial tiles and counters
    ("nvfp4", 128, 512, 4096, True, False),   # split-K through a cluster: status word only
    ("mxfp8", 2048, 2560, 512, False, False), # no split
    ("nvfp4", 300, 400, 608, True, False),    # ragged tiles
])
def test_noalloc_matches_plan_twice(kind, M, N, K, epi, workspace, monkeypatch):
    if workspace:
        monkeypatch.setenv("BSG_SPLIT_WORKSPACE", "1")
    prob = P.make_problem(kind, M, N, K)
    dp = P.DeviceProblem(prob, out="bf16", bias=epi, silu=epi)
    with dp.plan() as plan:
        plan.run()
        plan.check_status()
        want = dp.result()
    _, abs_sum = P.reference(prob, "bf16", dp.bias_vals, epi)
    for _ in range(2):
        got = _call_noalloc(dp, prob)
        tol = R.tolerance(want, got, abs_sum, prob["alpha"], epi, "bf16")
        assert np.all(np.abs(got - want) <= tol)
    P.assert_parity(got, prob, "bf16", dp.bias_vals, epi)


def test_noalloc_rejects_problems_beyond_its_scratch(monkeypatch):
    # 64 splits x 4 tiles x 64 KiB of partials = 16 MiB, beyond the 16 MiB array once the
    # counters are added
    monkeypatch.setenv("BSG_FORCE_BN", "128")
    monkeypatch.setenv("BSG_FORCE_SPLITS", "64")
    monkeypatch.setenv("BSG_SPLIT_WORKSPACE", "1")
    prob = P.make_problem("nvfp4", 128, 512, 16384)
    dp = P.DeviceProblem(prob)
    with pytest.raises(bsg.BsgError) as e:
        bsg.bsg_gemm_noalloc(bsg.BSG_NVFP4, bsg.BSG_OUT_BF16, 128, 512, 16384, dp.A, dp.B, dp.SFA, dp.SFB, dp.D,
                             alpha=float(prob["alpha"]))
    assert e.value.name == "BSG_ERR_SHAPE"
    assert "scratch" in str(e.value)
