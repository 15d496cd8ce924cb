"""The C-ABI library builds, loads and exports every entry point its header declares;
host-side validation rejects bad arguments before touching a device (runs without a GPU)."""

import ctypes
import os
import re

import pytest

import fp4_gemm_blackwell_gb300 as bsg
from fp4_gemm_blackwell_gb300 import build as B

HEADER = os.path.join(B.INCLUDE, "bsgemm.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return bsg.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for want in ["bsg_plan_create", "bsg_plan_run", "bsg_plan_destroy", "bsg_plan_check_status",
                 "mxfp8_gemm", "nvfp4_gemm", "bsg_sf_bytes", "bsg_quantize", "bsg_quantize_bf16", "bsg_last_error",
                 "bsg_plan_run_operands"]:
        assert want in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version_and_sf_bytes(L):
    assert "sm_103a" in bsg.bsg_version()
    # rows padded to 128, scale columns to 4 (MXFP8 block 32, NVFP4 block 16)
    assert bsg.bsg_sf_bytes(bsg.BSG_MXFP8, 256, 256) == 256 * 8
    assert bsg.bsg_sf_bytes(bsg.BSG_MXFP8, 8000, 8192) == 8064 * 256
    assert bsg.bsg_sf_bytes(bsg.BSG_NVFP4, 8000, 8192) == 8064 * 512
    assert bsg.bsg_sf_bytes(bsg.BSG_NVFP4, 1, 32) == 128 * 4
    assert bsg.bsg_sf_bytes(bsg.BSG_MXFP8, 1, 160) == 128 * 8
    assert bsg.bsg_sf_bytes(bsg.BSG_MXFP8, 0, 32) == 0
    assert bsg.bsg_sf_bytes(bsg.BSG_MXFP8, 4, 48) == 0
    assert bsg.bsg_sf_bytes(bsg.BSG_NVFP4, 300, 272) == 384 * 20   # an NVFP4 output's N: 17 blocks
    assert bsg.bsg_sf_bytes(bsg.BSG_NVFP4, 4, 40) == 0
    assert bsg.bsg_sf_bytes(7, 4, 64) == 0


def _plan_status(L, **kw):
    base = dict(kind=0, out=1, flags=0, M=128, N=128, K=128, A=16, B=32, SFA=48, SFB=64, bias=None,
                D=80, alpha=1.0, alpha_dev=None, C=None, beta=0.0, alpha_row=None, alpha_col=None, batches=0,
                strides=(0, 0, 0, 0, 0, 0), group_index=None, SFD=None, d_scale=None)
    base.update(kw)
    d = bsg.BsgDesc(base["kind"], base["out"], base["flags"], base["M"], base["N"], base["K"], base["A"],
                    base["B"], base["SFA"], base["SFB"], base["bias"], base["D"], base["alpha"], base["alpha_dev"],
                    base["C"], base["beta"], base["alpha_row"], base["alpha_col"], base["batches"], *base["strides"],
                    base["group_index"], base["SFD"], base["d_scale"])
    h = ctypes.c_void_p()
    st = L.bsg_plan_create(ctypes.byref(h), ctypes.byref(d))
    assert h.value is None
    return st


@pytest.mark.parametrize("kw,status", [
    (dict(kind=5), 1), (dict(out=3), 5), (dict(flags=8), 1),
    (dict(M=0), 2), (dict(N=8), 2), (dict(N=120), 2), (dict(K=48), 2), (dict(K=16), 2),
    (dict(M=1 << 21), 2), (dict(A=None), 1), (dict(D=None), 1), (dict(flags=1), 1),
    (dict(flags=4), 1), (dict(A=24), 3), (dict(SFB=72), 3), (dict(flags=1, bias=88), 3),
    (dict(flags=128), 1), (dict(flags=8, C=104), 3), (dict(flags=16), 1), (dict(flags=32), 1),
    (dict(flags=16, alpha_row=130), 3), (dict(flags=32, alpha_col=6), 3),
    # batched: L out of range; a stride below one entry; a stride not a multiple of 16
    (dict(batches=-1), 2), (dict(batches=70000), 2),
    (dict(batches=2, strides=(0, 16384, 2048, 2048, 32768, 0)), 2),
    (dict(batches=2, strides=(16384 + 8, 16384, 2048, 2048, 32768, 0)), 2),
    (dict(batches=2, strides=(16384, 16384, 2048, 2048, 32768 - 16, 0)), 2),
    # grouped: no groups; no group_index; a misaligned group_index; a B stride below one expert
    (dict(flags=64), 2), (dict(flags=64, batches=4), 1), (dict(flags=64, batches=4, group_index=6), 3),
    (dict(flags=64, batches=4, group_index=256, strides=(0, 16384 - 16, 0, 2048, 0, 0)), 2),
    (dict(flags=64, batches=4, group_index=256, strides=(0, 16384, 0, 512 - 16, 0, 0)), 2),
    # NVFP4 output: an unknown output type; no SFD or d_scale; a misaligned SFD or d_scale;
    # batches or groups with it
    (dict(out=3), 5), (dict(out=2), 1), (dict(out=2, SFD=96), 1), (dict(out=2, d_scale=100), 1),
    (dict(out=2, SFD=104, d_scale=100), 3), (dict(out=2, SFD=96, d_scale=102), 3),
    (dict(out=2, SFD=96, d_scale=100, batches=2, strides=(16384, 16384, 512, 512, 16384, 0)), 2),
    (dict(out=2, SFD=96, d_scale=100, flags=64, batches=2, group_index=256, strides=(0, 16384, 0, 512, 0, 0)), 2),
])
def test_invalid_descriptors_are_rejected_before_device_work(L, kw, status):
    assert _plan_status(L, **kw) == status
    assert bsg.bsg_last_error() != ""


def test_null_handles(L):
    assert L.bsg_plan_create(None, None) == 1
    assert L.bsg_plan_run(None, None) == 1
    assert L.bsg_plan_run_operands(None, None, None) == 1
    assert L.bsg_plan_destroy(None) == 1
    assert L.bsg_plan_check_status(None) == 1
    assert L.bsg_plan_variant(None) == b""
    with pytest.raises(bsg.BsgError) as e:
        bsg.bsg_plan_run(None, 0)
    assert e.value.name == "BSG_ERR_INVALID_ARG"


@pytest.mark.parametrize("args,status", [
    ((7, 16, 128, 128, 32, 48, 64), 1),        # kind
    ((0, 16, 0, 128, 32, 48, 64), 2),          # rows
    ((0, 16, 128, 48, 32, 48, 64), 2),         # K % 32
    ((0, None, 128, 128, 32, 48, 64), 1),      # null x
    ((1, 16, 128, 128, 32, 48, None), 1),      # NVFP4 needs global_scale
    ((0, 20, 128, 128, 32, 48, 64), 3),        # misaligned x
])
def test_quantize_validation(L, args, status):
    kind, x, rows, K, codes, sf, gs = args
    assert L.bsg_quantize(kind, x, rows, K, codes, sf, gs, None) == status
    assert L.bsg_quantize_bf16(kind, x, rows, K, codes, sf, gs, None) == status


@pytest.mark.parametrize("args,status", [
    ((None, 0, 128, 256, 32, 48, 64), 1),      # null x
    ((16, 0, 128, 256, 32, 48, None), 1),      # null global scale
    ((16, 1, 0, 256, 32, 48, 64), 2),          # rows < 1
    ((16, 0, 128, 48, 32, 48, 64), 2),         # K not a multiple of 32
    ((24, 0, 128, 256, 32, 48, 64), 3),        # x not 16-byte aligned
    ((16, 1, 128, 256, 32, 48, 66), 3),        # global scale not 4-byte aligned
])
def test_quantize_given_scale_validation(L, args, status):
    x, bf16, rows, K, codes, sf, gs = args
    assert L.bsg_quantize_nvfp4_scaled(x, bf16, rows, K, codes, sf, gs, None) == status


def test_one_shot_validation(L):
    # N not a multiple of 16 and a device alpha through the host-alpha call are refused
    assert L.mxfp8_gemm(16, 32, 48, 64, 80, ctypes.c_float(1.0), 128, 120, 128, 1, None) == 2
    assert L.nvfp4_gemm(16, 32, 48, 64, 80, None, ctypes.c_float(1.0), 4, 128, 128, 128, 1, None) == 1


def test_python_structures_match_the_header_layout():
    # bsg_desc and bsg_operands as the C compiler lays them out from include/bsgemm.h (a probe
    # built with gcc under the git-ignored _build/) against the ctypes structures of the binding:
    # the same size and every field at the same offset, so that appended fields cannot drift.
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = os.path.join(root, "_build", "abi_layout")
    os.makedirs(out, exist_ok=True)
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "bsgemm.h"', "int main(void) {"]
    for cname, py in (("bsg_desc", bsg.BsgDesc), ("bsg_operands", bsg.BsgOperands)):
        lines.append('  printf("%s %%zu\\n", sizeof(%s));' % (cname, cname))
        for field, _ in py._fields_:
            lines.append('  printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (cname, field, cname, field))
    lines += ["  return 0;", "}"]
    src = os.path.join(out, "layout.c")
    exe = os.path.join(out, "layout")
    with open(src, "w") as f:
        f.write("\n".join(lines) + "\n")
    subprocess.run([gcc, "-std=c11", "-I", os.path.join(root, "include"), src, "-o", exe], check=True)
    got = dict(line.split() for line in subprocess.run([exe], check=True, capture_output=True,
                                                       text=True).stdout.splitlines())
    for cname, py in (("bsg_desc", bsg.BsgDesc), ("bsg_operands", bsg.BsgOperands)):
        assert int(got[cname]) == ctypes.sizeof(py), cname
        for field, _ in py._fields_:
            assert int(got["%s.%s" % (cname, field)]) == getattr(py, field).offset, (cname, field)


def test_allocation_free_entry_points_validate_before_device_work(L):
    # a bad descriptor is refused by the allocation-free call as by plan creation; without a GPU
    # the status query reports a CUDA error instead of crashing
    d = bsg.BsgDesc(0, 1, 0, 128, 120, 128, 16, 32, 48, 64, None, 80, 1.0, None, None, 0.0, None, None, 0,
                    0, 0, 0, 0, 0, 0, None, None, None)
    assert L.bsg_gemm_noalloc(ctypes.byref(d), None) == 2          # N not a multiple of 16
    assert L.bsg_gemm_noalloc(None, None) == 1
    st = L.bsg_noalloc_check_status(None)
    assert st in (0, 6, 7)                                          # OK / not sm_103 / CUDA error
