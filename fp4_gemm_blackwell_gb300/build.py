"""In-tree build of libbsgemm.so (CUDA kernels + C ABI) for sm_103a with nvcc.

Objects go to ``_build/<machine>/`` at the repository root, the library next to this
file.  Translation units compile in parallel; a unit is rebuilt when it or any header
of the library is newer than its object.
"""

import glob
import os
import platform
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libbsgemm.so")
# Programs built beside the library (csrc/*_main.cu, linked against it): the native
# launch-overhead loop that bench.py runs.
LAUNCH_LOOP = os.path.join(PKG, "bsg_launch_loop")
# Test-only probe kernels (tests/csrc/*.cu), each built into its own shared library beside its
# source; only the GPU tests load them.
TEST_CSRC = os.path.join(ROOT, "tests", "csrc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-I" + INCLUDE, "-I" + CSRC,
          "-Xcompiler", "-fPIC,-fvisibility=hidden"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _newest(paths):
    return max((os.path.getmtime(p) for p in paths), default=0.0)


def build(verbose=False, force=False):
    """Compile every .cu under csrc/ and link libbsgemm.so; returns the library path."""
    nvcc = _nvcc()
    objdir = os.path.join(ROOT, "_build", platform.machine())
    os.makedirs(objdir, exist_ok=True)
    sources = sorted(f for f in glob.glob(os.path.join(CSRC, "*.cu")) if not f.endswith("_main.cu"))
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    hdr_time = _newest(headers)
    procs, objs = [], []
    for src in sources:
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_time):
            continue
        cmd = [nvcc] + ARCH + CFLAGS + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append("%s:\n%s" % (src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    if force or procs or not os.path.exists(LIB) or os.path.getmtime(LIB) < _newest(objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-Xlinker", "--exclude-libs=ALL"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(tmp, LIB)
    main_src = os.path.join(CSRC, "launch_loop_main.cu")
    if force or not os.path.exists(LAUNCH_LOOP) or os.path.getmtime(LAUNCH_LOOP) < max(
            os.path.getmtime(LIB), os.path.getmtime(main_src)):
        cmd = [nvcc] + ARCH + ["-O3", "-std=c++17", "-I" + INCLUDE, "-o", LAUNCH_LOOP, main_src, "-L" + PKG,
                               "-lbsgemm", "-Xlinker", "-rpath,$ORIGIN"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("launch loop build failed:\n" + r.stdout.decode(errors="replace"))
    for src in sorted(glob.glob(os.path.join(TEST_CSRC, "*.cu"))):
        so = os.path.join(TEST_CSRC, "lib" + os.path.basename(src)[:-3] + ".so")
        if not force and os.path.exists(so) and os.path.getmtime(so) >= max(os.path.getmtime(src), hdr_time):
            continue
        cmd = [nvcc] + ARCH + CFLAGS + ["-shared", "-o", so, src]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("test probe build failed:\n" + r.stdout.decode(errors="replace"))
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
