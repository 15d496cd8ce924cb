"""The allocation-free GEMM entry point against the plan entry point.

bsg_gemm_noalloc is for callers that may not allocate device memory when they run a GEMM
(allocator callbacks, engines with a fixed device-memory budget); it keeps its scratch in a
static device array instead of a plan's workspace.  Here it is called through the C ABI twice
in a row per problem and each output is compared with bsg_plan_run's output on the same
operands, within the parity tolerance the other GEMM tests use; once warmed up, its calls must
leave the device's free memory and the caching allocator's counters as they were; a bounded
wait that runs out must be reported by bsg_noalloc_check_status.  This file is collected last.
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


def test_noalloc_allocates_nothing_after_first_use():
    # first use of the shape loads the kernel and the scratch array (outside the measured part)
    prob = P.make_problem("nvfp4", 128, 512, 4096)
    dp = P.DeviceProblem(prob, out="bf16", bias=True, silu=True)
    want = _call_noalloc(dp, prob)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for _ in range(5):
        bsg.bsg_gemm_noalloc(bsg.BSG_NVFP4, bsg.BSG_OUT_BF16, 128, 512, 4096, dp.A, dp.B, dp.SFA, dp.SFB, dp.D,
                             alpha=float(prob["alpha"]), flags=dp.flags, bias=dp.bias)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0, "device free memory changed by %d bytes" % (free0 - free1)
    for k in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
        assert stats1.get(k, 0) == stats0.get(k, 0), k
    bsg.bsg_noalloc_check_status()
    assert np.array_equal(dp.result(), want)


def test_noalloc_wait_timeout_is_reported_then_cleared():
    # the test hook makes every producer leave its first stage unfilled, with a 50 ms wait limit:
    # the kernel gives up and records it in the scratch array's status word, which the status
    # query reports once and clears; the next call, without the hook, matches the plan's result
    prob = P.make_problem("mxfp8", 256, 256, 256)
    dp = P.DeviceProblem(prob)
    with dp.plan() as plan:
        plan.run()
        plan.check_status()
        want = dp.result()
    bsg.bsg_noalloc_check_status()
    try:
        bsg.bsg_plan_debug_set(None, 1, 50_000_000)
        _call_noalloc(dp, prob)
        with pytest.raises(bsg.BsgError) as e:
            bsg.bsg_noalloc_check_status()
        assert e.value.name == "BSG_ERR_DEVICE_TIMEOUT"
        bsg.bsg_noalloc_check_status()   # cleared by the query that reported it
    finally:
        bsg.bsg_plan_debug_set(None, 0, 0)
    got = _call_noalloc(dp, prob)
    bsg.bsg_noalloc_check_status()
    assert np.array_equal(got, want)
