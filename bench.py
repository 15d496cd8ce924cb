"""Benchmark of the block-scaled GEMM library on GB300.

Headline workload (one step = one GEMM through the library's plan, operands already
quantised and resident in HBM):
    NVFP4 GEMM M=N=K=8192, BF16 bias + SiLU, BF16 out (tensor-bound: the configuration the
    pages' "% of dense block-scaled tensor peak" target is stated at).
Metric: block-scaled GEMM TFLOPS (2*M*N*K per step) and its fraction of the FP4 tensor peak;
the same JSON line gives the host microseconds per call against the kernel time, the end-to-end
number through the C ABI with host buffers, the other workloads (the skinny-M HBM-bound NVFP4
128x4096x4096 with its HBM roofline, MXFP8 256^3, MXFP8 8192^3 FP16/BF16, NVFP4
8000x8192x8192, the launch loop, ...) and the CPU oracle timed on this machine's host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--quick]

Inputs rotate over copies whose bytes together exceed the 129 MB L2 (for the headline: two
copies of 75 MB of operands and a 134 MB output each), so a step's operands are not in L2 from
the previous use.  Timed regions are bracketed by torch.cuda.synchronize (and a barrier with
N > 1) and measured with CUDA events on the stream the kernels are launched on.
"""

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

MH, NH, KH = 8192, 8192, 8192         # the headline workload (NVFP4, bias + SiLU, BF16 out)
M1, N1, K1 = 128, 4096, 4096          # the skinny-M workload (HBM-bound)
L2_BYTES = 129 * 1024 * 1024
SM_COUNT_DEFAULT = 152


# ---------------------------------------------------------------- peaks and clocks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# dense tensor rate of each operand type relative to bf16 (nominal GB300: bf16 2.25, fp8 4.5, fp4 13.5 PF)
NOMINAL_RATIO = {"fp8": 4.5 / 2.25, "fp4": 13.5 / 2.25}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while a region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, path=None):
        """path: where the raw samples go (BSG_CLOCKS_CSV, else a temporary file)."""
        self.index = index
        self.proc = None
        self.path = path or os.environ.get("BSG_CLOCKS_CSV") or os.path.join(
            tempfile.gettempdir(), "bsg_clocks_%d_%d.csv" % (os.getpid(), index))

    def start(self):
        try:
            os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, watts, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            t = [x.strip() for x in line.split(",")]
            if len(t) < 8:
                continue
            try:
                sm.append(float(t[0]))
                smax.append(float(t[1]))
            except ValueError:
                continue
            try:
                watts.append(float(t[2]))
            except ValueError:
                pass
            for n, v in zip(names, t[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "power_w": statistics.median(watts) if watts else None, "samples": len(sm)}


def strip_comments(src):
    """C++ source without its // and /* */ comments or blank lines (string literals in these
    files hold PTX, which has no comment markers): edits to comments leave the hash alone."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_hash():
    """Hash of the kernels' code (comments ignored), the key under which profiles/traffic.json
    records DRAM traffic: a record whose hash differs was taken of other code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp4_gemm_blackwell_gb300", "csrc")
    for name in ("gemm_kernel.cuh", "gemm_pair_kernel.cuh", "nvfp4_codec.cuh", "ptx.cuh", "bsg_internal.h"):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """dram read+write bytes per launch from a committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel + "|" + workload]
    except Exception:
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- operands
class Operands:
    """One quantised operand on the device, made by the library's own quantiser."""

    def __init__(self, bsg, kind, rows, K, seed):
        from fp4_gemm_blackwell_gb300 import synth
        gen = synth.normal if kind == "mxfp8" else synth.normal_rowscaled
        x = torch.from_numpy(gen(rows, K, seed)).cuda()
        k = bsg.BSG_MXFP8 if kind == "mxfp8" else bsg.BSG_NVFP4
        self.codes = torch.empty(rows * K if kind == "mxfp8" else rows * K // 2, dtype=torch.uint8, device="cuda")
        self.sf = torch.empty(bsg.bsg_sf_bytes(k, rows, K), dtype=torch.uint8, device="cuda")
        gs = torch.zeros(1, dtype=torch.float32, device="cuda")
        bsg.bsg_quantize(k, x, rows, K, self.codes, self.sf, gs)
        torch.cuda.synchronize()
        self.s = float(gs.item()) if kind == "nvfp4" else 1.0
        del x

    def clone(self):
        c = Operands.__new__(Operands)
        c.codes, c.sf, c.s = self.codes.clone(), self.sf.clone(), self.s
        return c


def algorithmic_bytes(kind, M, N, K, bias=False, residual=False, factors=False, L=1):
    """Bytes one launch must move at least: codes + padded scales of A and B, the 16-bit output,
    and the bias, C and factor vectors when used (L entries of everything but the bias and
    factors, which the entries share)."""
    cb = 1 if kind == "mxfp8" else 0.5
    blk = 32 if kind == "mxfp8" else 16
    sf = lambda rows: ((rows + 127) // 128 * 128) * ((K // blk + 3) // 4 * 4)
    b = L * (M * K * cb + N * K * cb + sf(M) + sf(N) + M * N * 2)
    if bias:
        b += N * 2
    if residual:
        b += L * M * N * 2
    if factors:
        b += (M + N) * 4
    return int(b)


class Problem:
    """R device copies of one GEMM problem (operands, bias, output) with a plan per copy."""

    def __init__(self, bsg, kind, M, N, K, out="bf16", bias=False, silu=False, copies=1, seeds=(0, 1),
                 residual=False, factors=False, L=1):
        """residual: beta * C from a separate M x N matrix per copy (beta = 1); factors: per-row
        and per-column alpha vectors (U(0.5, 2)); L > 1: a batch of L problems of this shape per
        copy, entry l being rows l*M.. of one (L*M) x K operand A (likewise B), quantised as one
        tensor (M and N multiples of 128, so every entry's scales start on a band)."""
        from fp4_gemm_blackwell_gb300 import synth
        self.kind, self.M, self.N, self.K, self.out, self.L = kind, M, N, K, out, L
        self.residual, self.factors = residual, factors
        if L > 1 and (M % 128 or N % 128):
            raise ValueError("batched problems here need M and N multiples of 128")
        a = Operands(bsg, kind, L * M, K, seeds[0])
        b = Operands(bsg, kind, L * N, K, seeds[1])
        self.alpha = float(np.float32(np.float32(a.s) * np.float32(b.s)))
        self.flags = ((bsg.BSG_F_BIAS if bias else 0) | (bsg.BSG_F_SILU if silu else 0) |
                      (bsg.BSG_F_C if residual else 0) | (bsg.BSG_F_ALPHA_ROW | bsg.BSG_F_ALPHA_COL if factors else 0))
        self.extra = []
        cbits = synth.bias(L * M * N, seed=5, std=1.0, out=out)[0] if residual else None
        cb = 1 if kind == "mxfp8" else 2
        strides = dict(stride_A=M * K // cb, stride_B=N * K // cb, stride_SFA=bsg.bsg_sf_bytes(
            self._k(bsg), M, K), stride_SFB=bsg.bsg_sf_bytes(self._k(bsg), N, K), stride_D=2 * M * N,
            stride_C=2 * M * N if residual else 0)
        g = torch.Generator(device="cpu")
        g.manual_seed(6)
        ar = (torch.rand(M, generator=g) * 1.5 + 0.5).cuda() if factors else None
        ac = (torch.rand(N, generator=g) * 1.5 + 0.5).cuda() if factors else None
        bias_t = None
        if bias:
            bits, _ = synth.bias(N, out=out)
            bias_t = torch.from_numpy(bits.view(np.int16)).cuda()
        out_t = bsg.BSG_OUT_BF16 if out == "bf16" else bsg.BSG_OUT_F16
        k = bsg.BSG_MXFP8 if kind == "mxfp8" else bsg.BSG_NVFP4
        self.sets, self.plans = [], []
        for i in range(copies):
            ai, bi = (a, b) if i == 0 else (a.clone(), b.clone())
            bt = None if bias_t is None else (bias_t if i == 0 else bias_t.clone())
            d = torch.empty(L * M * N, dtype=torch.int16, device="cuda")
            c = torch.from_numpy(cbits.view(np.int16)).cuda() if residual else None
            self.extra.append(c)
            self.sets.append((ai, bi, bt, d))
            self.plans.append(bsg.Plan(k, out_t, M, N, K, ai.codes, bi.codes, ai.sf, bi.sf, d,
                                       alpha=self.alpha, flags=self.flags, bias=bt, C=c, beta=1.0,
                                       alpha_row=ar, alpha_col=ac, L=L if L > 1 else 0,
                                       strides=strides if L > 1 else None))
        self.variant = self.plans[0].variant

    def _k(self, bsg):
        return bsg.BSG_MXFP8 if self.kind == "mxfp8" else bsg.BSG_NVFP4

    def flops(self):
        return 2.0 * self.M * self.N * self.K * self.L

    def algorithmic_bytes(self):
        return algorithmic_bytes(self.kind, self.M, self.N, self.K, bias=bool(self.flags & 1),
                                 residual=self.residual, factors=self.factors, L=self.L)

    def close(self):
        for p in self.plans:
            p.close()
        self.plans = []


def copies_to_exceed_l2(bytes_per_copy):
    return max(1, min(64, int(np.ceil(1.5 * L2_BYTES / max(bytes_per_copy, 1)))))


def graph_time(plans, steps, warmup, barrier=None):
    """Capture `steps` launches (rotating over plans) in one CUDA graph and time one replay.

    Returns (elapsed_ms, number of our kernel launches in the timed region)."""
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(warmup):
            plans[i % len(plans)].run(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(steps):
            plans[i % len(plans)].run(stream)
    with torch.cuda.stream(stream):
        g.replay()                                   # one untimed replay (warm graph upload)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    ms = start.elapsed_time(end)
    del g
    return ms, steps


def stream_time(plans, steps, warmup):
    """Plain stream launches behind a device-side sleep, so that the queue is full when the
    timed region starts: the events then measure back-to-back kernel execution."""
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(warmup):
            plans[i % len(plans)].run(stream)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(2e6) * max(1, steps // 50))
        start.record(stream)
        t0 = time.perf_counter()
        for i in range(steps):
            plans[i % len(plans)].run(stream)
        host_s = time.perf_counter() - t0
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end), host_s * 1e6 / steps


# ---------------------------------------------------------------- the headline step
def headline(bsg, steps, warmup, barrier):
    """The headline GEMM, two operand / output copies (420 MB together, above the L2) in turn."""
    prob = Problem(bsg, "nvfp4", MH, NH, KH, bias=True, silu=True, copies=2)
    ms, launches = graph_time(prob.plans, steps, warmup, barrier)
    stream_ms, host_us = stream_time(prob.plans, min(steps, 1000), warmup)
    return dict(problem=prob, ms=ms, launches=launches, copies=2, per_copy=prob.algorithmic_bytes(),
                stream_kernel_us=stream_ms * 1e3 / min(steps, 1000), host_us_per_run=host_us)


def skinny_headline(bsg, peaks, steps=400, warmup=10):
    """NVFP4 128 x 4096 x 4096 with bias + SiLU (skinny M, HBM-bound), inputs rotated over enough
    copies to exceed L2: kernel time, host time per plan run and the HBM roofline."""
    probe = Problem(bsg, "nvfp4", M1, N1, K1, bias=True, silu=True, copies=1)
    per_copy = probe.algorithmic_bytes()
    probe.close()
    copies = copies_to_exceed_l2(per_copy)
    prob = Problem(bsg, "nvfp4", M1, N1, K1, bias=True, silu=True, copies=copies)
    ms, _ = graph_time(prob.plans, steps, warmup)
    stream_ms, host_us = stream_time(prob.plans, min(steps, 1000), warmup)
    us = ms * 1e3 / steps
    gbs = per_copy / (us * 1e-6) / 1e9
    r = {"us": round(us, 3), "tflops": round(prob.flops() / (us * 1e-6) / 1e12, 1), "variant": prob.variant,
         "l2": "inputs rotate over %d copies (%.0f MB > 129 MB L2)" % (copies, copies * per_copy / 2 ** 20),
         "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": round(gbs / peaks["hbm_gbs"], 4),
                      "traffic": recorded_traffic("bsg_gemm_kernel<nvfp4,%s>" % prob.variant.split("_")[1],
                                                  "nvfp4_m128_n4096_k4096"),
                      "algorithmic_bytes_per_launch": per_copy,
                      "peak_source": peaks["source"] + " hbm_gbs (burst copy)"},
         "host_us_per_plan_run": round(host_us, 3), "kernel_us_stream_back_to_back": round(stream_ms * 1e3 / min(
             steps, 1000), 3)}
    prob.close()
    return r


def e2e(bsg, steps, M=MH, N=NH, K=KH):
    """The workload through the one-shot C-ABI call, host buffers in and out every step: each
    step copies its A, SFA, B, SFB and bias from pinned host memory (one copy: the five inputs
    sit at 256-byte-aligned offsets of one block), runs nvfp4_gemm and copies D back to pinned
    host memory.  Steps are pipelined the way a serving loop would run them: two device buffer
    sets, the copy in (copy stream), the GEMM (compute stream) and the copy out (a third stream)
    of consecutive steps overlap; every copy of every step is inside the timed region."""
    prob = Problem(bsg, "nvfp4", M, N, K, bias=True, silu=True, copies=1)
    a0, b0, bias0, d0 = prob.sets[0]
    parts = [a0.codes, a0.sf, b0.codes, b0.sf, bias0]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_blob = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(parts, offs):
        n = t.numel() * t.element_size()
        host_blob[o:o + n].copy_(t.view(torch.uint8).reshape(-1).cpu())
    alpha, flags = prob.alpha, prob.flags
    prob.close()
    sets = [(torch.empty(total, dtype=torch.uint8, device="cuda"), torch.empty_like(d0)) for _ in range(2)]
    d_host = [torch.empty_like(d0, device="cpu").pin_memory() for _ in sets]
    h2d = sum(t.numel() * t.element_size() for t in parts)
    d2h = d0.numel() * d0.element_size()
    L = bsg.lib()
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = [{k: torch.cuda.Event() for k in ("in", "comp", "out")} for _ in sets]
    for e in ev:  # a buffer set starts free
        for k in ("comp", "out"):
            e[k].record(s_comp)

    def step(j):
        i = j % len(sets)
        blob, d = sets[i]
        base = blob.data_ptr()
        s_in.wait_event(ev[i]["comp"])           # the GEMM that last read this set is done
        with torch.cuda.stream(s_in):
            blob.copy_(host_blob, non_blocking=True)
        ev[i]["in"].record(s_in)
        s_comp.wait_event(ev[i]["in"])
        s_comp.wait_event(ev[i]["out"])          # this set's previous result has left the GPU
        st = L.nvfp4_gemm(d.data_ptr(), base + offs[0], base + offs[2], base + offs[1], base + offs[3],
                          base + offs[4], alpha, flags, M, N, K, bsg.BSG_OUT_BF16, s_comp.cuda_stream)
        if st != 0:
            raise bsg.BsgError(st, bsg.bsg_last_error())
        ev[i]["comp"].record(s_comp)
        s_out.wait_event(ev[i]["comp"])
        with torch.cuda.stream(s_out):
            d_host[i].copy_(d, non_blocking=True)
        ev[i]["out"].record(s_out)

    for j in range(6):
        step(j)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for j in range(steps):
        step(j)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    bsg.bsg_cache_clear()
    tflops = 2.0 * M * N * K * steps / dt / 1e12
    return {"value": round(tflops, 4), "unit": "TFLOPS", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(dt * 1e3 / steps, 4), "steps": steps,
            "h2d_gbs": round(h2d * steps / dt / 1e9, 1),
            "path": "nvfp4_gemm (C ABI, cached plan) + one pinned H2D of A/SFA/B/SFB/bias + D2H of D; "
                    "consecutive steps overlapped on three streams with two device buffer sets"}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return rank, world, local, dist
    torch.cuda.set_device(0)
    return 0, 1, 0, None


def whole_job(ms_local, flops_per_step, steps, world, dist=None, device="cuda"):
    """The timed region's maximum over ranks (ms) and the whole-job throughput in TFLOPS: every
    rank's `steps` steps of `flops_per_step`, over that maximum."""
    ms_max = ms_local
    if dist is not None:
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_max = float(t.item())
    return ms_max, flops_per_step * steps * world / (ms_max * 1e-3) / 1e12


# ---------------------------------------------------------------- the other workloads
def tensor_peak(peaks, kind):
    return peaks["bf16_tflops"] * NOMINAL_RATIO["fp8" if kind == "mxfp8" else "fp4"]


def big_config(bsg, peaks, kind, M, N, K, out, bias, silu, steps=20, warmup=3, residual=False, factors=False):
    prob = Problem(bsg, kind, M, N, K, out=out, bias=bias, silu=silu, copies=1, residual=residual, factors=factors)
    ms, _ = graph_time(prob.plans, steps, warmup)
    us = ms * 1e3 / steps
    tf = prob.flops() / (us * 1e-6) / 1e12
    peak = tensor_peak(peaks, kind)
    r = {"us": round(us, 2), "tflops": round(tf, 1), "peak_tflops": round(peak, 1),
         "frac_of_peak": round(tf / peak, 4), "variant": prob.variant,
         "l2": "single input set of %.0f MB" % (prob.algorithmic_bytes() / 2 ** 20)}
    prob.close()
    return r


def skinny_config(bsg, peaks, steps=400, warmup=10, **epi):
    """The headline shape (NVFP4 128 x 4096 x 4096, bias + SiLU) with extra epilogue terms,
    inputs rotated over enough copies to exceed L2; kernel time and HBM roofline fraction."""
    p1 = Problem(bsg, "nvfp4", M1, N1, K1, bias=True, silu=True, copies=1, **epi)
    cp = copies_to_exceed_l2(p1.algorithmic_bytes())
    p1.close()
    prob = Problem(bsg, "nvfp4", M1, N1, K1, bias=True, silu=True, copies=cp, **epi)
    ms, _ = graph_time(prob.plans, steps, warmup)
    us = ms * 1e3 / steps
    gbs = prob.algorithmic_bytes() / (us * 1e-6) / 1e9
    r = {"us": round(us, 3), "tflops": round(prob.flops() / (us * 1e-6) / 1e12, 1), "gbs": round(gbs, 1),
         "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": prob.algorithmic_bytes(),
         "variant": prob.variant}
    prob.close()
    return r


def batched_config(bsg, peaks, L, steps=200, warmup=10):
    """L problems of the headline shape (NVFP4 128 x 4096 x 4096, bias + SiLU) in one launch,
    inputs rotated over enough copies to exceed L2."""
    p1 = Problem(bsg, "nvfp4", M1, N1, K1, bias=True, silu=True, copies=1, L=L)
    cp = copies_to_exceed_l2(p1.algorithmic_bytes())
    p1.close()
    prob = Problem(bsg, "nvfp4", M1, N1, K1, bias=True, silu=True, copies=cp, L=L)
    ms, _ = graph_time(prob.plans, steps, warmup)
    us = ms * 1e3 / steps
    gbs = prob.algorithmic_bytes() / (us * 1e-6) / 1e9
    r = {"L": L, "us": round(us, 3), "us_per_entry": round(us / L, 3),
         "tflops": round(prob.flops() / (us * 1e-6) / 1e12, 1), "gbs": round(gbs, 1),
         "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "variant": prob.variant, "copies": cp}
    prob.close()
    return r


MOE_TOKENS = (97, 211, 64, 150, 128, 30, 180, 164)  # rows routed to each of 8 experts (1024 in all)


def grouped_config(bsg, peaks, steps=200, warmup=10):
    """Expert GEMMs of a mixture-of-experts layer: 8 groups (experts) of NVFP4 N=4096 x K=4096
    weights, MOE_TOKENS rows each in the 128-row-aligned grouped layout (group_index on the
    device, per-expert alpha_dev), bias + SiLU, BF16 out; one grouped launch per step, and for
    comparison the same 8 problems as 8 plain launches.  Inputs rotate over enough copies to
    exceed L2.  FLOPs and bytes count the routed rows only."""
    from fp4_gemm_blackwell_gb300 import synth
    G, N, K = len(MOE_TOKENS), N1, K1
    gidx = []
    for g, n in enumerate(MOE_TOKENS):
        gidx += [g] * n + [-1] * (-n % 128)
    M = len(gidx)
    rows = sum(MOE_TOKENS)
    cb = 2  # NVFP4: two elements per byte
    per_copy = M * K // cb + G * N * K // cb + M * N * 2
    cp = copies_to_exceed_l2(per_copy)
    k = bsg.BSG_NVFP4
    bits, _ = synth.bias(N, out="bf16")
    bias_t = torch.from_numpy(bits.view(np.int16)).cuda()
    gi = torch.tensor(gidx, dtype=torch.int32, device="cuda")
    grouped, separate, keep = [], [], []
    for i in range(cp):
        a = Operands(bsg, "nvfp4", M, K, 10 + i)
        b = Operands(bsg, "nvfp4", G * N, K, 20 + i)  # expert g: rows g*N.. of one operand
        alpha = float(np.float32(np.float32(a.s) * np.float32(b.s)))
        ad = torch.full((G,), alpha, dtype=torch.float32, device="cuda")
        d = torch.empty(M * N, dtype=torch.int16, device="cuda")
        keep += [a, b, ad, d]
        strides = dict(stride_B=N * K // cb, stride_SFB=bsg.bsg_sf_bytes(k, N, K))
        grouped.append(bsg.Plan(k, bsg.BSG_OUT_BF16, M, N, K, a.codes, b.codes, a.sf, b.sf, d,
                                flags=bsg.BSG_F_GROUPED | bsg.BSG_F_ALPHA_DEVICE | bsg.BSG_F_BIAS | bsg.BSG_F_SILU,
                                bias=bias_t, alpha_dev=ad, L=G, strides=strides, group_index=gi))
        row0 = 0
        for g, n in enumerate(MOE_TOKENS):  # the same rows as G plain problems
            ab = a.codes.view(M, K // cb)[row0:row0 + n]
            sfa = a.sf[row0 // 128 * bsg.bsg_sf_bytes(k, 128, K):]
            separate.append(bsg.Plan(k, bsg.BSG_OUT_BF16, n, N, K, ab, b.codes.view(G * N, K // cb)[g * N:],
                                     sfa, b.sf[g * bsg.bsg_sf_bytes(k, N, K):], d.view(M, N)[row0:],
                                     alpha=alpha, flags=bsg.BSG_F_BIAS | bsg.BSG_F_SILU, bias=bias_t))
            row0 += n + (-n % 128)
    ms, _ = graph_time(grouped, steps, warmup)
    us = ms * 1e3 / steps
    ms_s, _ = graph_time(separate, steps * G, warmup * G)
    us_s = ms_s * 1e3 / steps
    flops = 2.0 * rows * N * K
    nbytes = rows * K // cb + G * N * K // cb + bsg.bsg_sf_bytes(k, M, K) + G * bsg.bsg_sf_bytes(k, N, K) + \
        rows * N * 2 + N * 2 + 4 * G
    gbs = nbytes / (us * 1e-6) / 1e9
    r = {"groups": G, "rows": list(MOE_TOKENS), "N": N, "K": K, "us": round(us, 3),
         "tflops": round(flops / (us * 1e-6) / 1e12, 1), "gbs": round(gbs, 1),
         "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes,
         "variant": grouped[0].variant, "separate_launches_us": round(us_s, 3), "copies": cp}
    for pl in grouped + separate:
        pl.close()
    return r


class _OperandsRun:
    """plan.run_operands on one fixed buffer set, with the run(stream) method graph_time calls."""

    def __init__(self, plan, a, b, bias, d, alpha_dev):
        self.plan, self.args = plan, (a.codes, b.codes, a.sf, b.sf, d)
        self.kw = dict(bias=bias, alpha_dev=alpha_dev)

    def run(self, stream=None):
        self.plan.run_operands(*self.args, stream=stream, **self.kw)


def remap_config(bsg, peaks, steps=400, warmup=10):
    """The headline workload with ONE plan run on every input copy by bsg_plan_run_operands (its
    tensor maps rewritten on the device each launch), against one plan per copy."""
    p1 = Problem(bsg, "nvfp4", M1, N1, K1, bias=True, silu=True, copies=1)
    cp = copies_to_exceed_l2(p1.algorithmic_bytes())
    p1.close()
    prob = Problem(bsg, "nvfp4", M1, N1, K1, bias=True, silu=True, copies=cp)
    ms_plain, _ = graph_time(prob.plans, steps, warmup)
    ad = torch.tensor([prob.alpha], dtype=torch.float32, device="cuda")
    k = bsg.BSG_NVFP4
    a0, b0, bt0, d0 = prob.sets[0]
    one = bsg.Plan(k, bsg.BSG_OUT_BF16, M1, N1, K1, a0.codes, b0.codes, a0.sf, b0.sf, d0,
                   flags=prob.flags | bsg.BSG_F_ALPHA_DEVICE, bias=bt0, alpha_dev=ad)
    runs = [_OperandsRun(one, a, b, bt, d, ad) for (a, b, bt, d) in prob.sets]
    ms_remap, _ = graph_time(runs, steps, warmup)
    r = {"kernel_us_remap": round(ms_remap * 1e3 / steps, 3), "kernel_us_plans": round(ms_plain * 1e3 / steps, 3),
         "copies": cp, "variant": one.variant}
    one.close()
    prob.close()
    return r


def nvfp4_out_config(bsg, peaks, M, N, K, steps, warmup=5):
    """NVFP4 GEMM M x N x K with bias + SiLU whose output is NVFP4 (codes + swizzled scales, a
    device global scale): the form in which one layer's GEMM feeds the next.  Inputs rotate
    over enough copies to exceed L2; bytes count the NVFP4 output instead of a 16-bit one."""
    from fp4_gemm_blackwell_gb300 import synth
    k = bsg.BSG_NVFP4
    sfd_bytes = bsg.bsg_sf_bytes(k, M, N)
    one = M * K // 2 + N * K // 2 + bsg.bsg_sf_bytes(k, M, K) + bsg.bsg_sf_bytes(k, N, K) + M * N // 2 + sfd_bytes
    cp = copies_to_exceed_l2(one)
    bits, _ = synth.bias(N, out="bf16")
    bias_t = torch.from_numpy(bits.view(np.int16)).cuda()
    d_scale = torch.tensor([0.05], dtype=torch.float32, device="cuda")
    plans, keep = [], []
    for i in range(cp):
        a = Operands(bsg, "nvfp4", M, K, 30 + i)
        b = Operands(bsg, "nvfp4", N, K, 60 + i)
        d = torch.empty(M * N // 2, dtype=torch.uint8, device="cuda")
        sfd = torch.empty(sfd_bytes, dtype=torch.uint8, device="cuda")
        keep += [a, b, d, sfd]
        alpha = float(np.float32(np.float32(a.s) * np.float32(b.s)))
        plans.append(bsg.Plan(k, bsg.BSG_OUT_NVFP4, M, N, K, a.codes, b.codes, a.sf, b.sf, d, alpha=alpha,
                              flags=bsg.BSG_F_BIAS | bsg.BSG_F_SILU, bias=bias_t, SFD=sfd, d_scale=d_scale))
    ms, _ = graph_time(plans, steps, warmup)
    us = ms * 1e3 / steps
    tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
    gbs = (one + 2 * N) / (us * 1e-6) / 1e9
    r = {"us": round(us, 3), "tflops": round(tf, 1), "frac_of_fp4_peak": round(tf / tensor_peak(peaks, "nvfp4"), 4),
         "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": one + 2 * N,
         "variant": plans[0].variant, "copies": cp}
    for pl in plans:
        pl.close()
    return r


def l2_warm_config(bsg, peaks, steps=2000, warmup=20):
    """The headline workload with ONE input set, so that after the first launch its operands
    are L2-resident: the L2-warm number, reported beside the HBM-cold headline as context."""
    prob = Problem(bsg, "nvfp4", M1, N1, K1, bias=True, silu=True, copies=1)
    ms, _ = graph_time(prob.plans, steps, warmup)
    us = ms * 1e3 / steps
    r = {"us": round(us, 3), "tflops": round(prob.flops() / (us * 1e-6) / 1e12, 1), "l2": "warm (one input set)",
         "variant": prob.variant}
    prob.close()
    return r


def small_config(bsg, peaks, steps=2000, warmup=20):
    prob = Problem(bsg, "mxfp8", 256, 256, 256, copies=64)
    ms, _ = graph_time(prob.plans, steps, warmup)
    us = ms * 1e3 / steps
    tf = prob.flops() / (us * 1e-6) / 1e12
    r = {"us": round(us, 3), "tflops": round(tf, 2), "frac_of_peak": round(tf / tensor_peak(peaks, "mxfp8"), 5),
         "variant": prob.variant, "l2": "64 rotating sets, L2-resident (17 MB)", "bound": "launch latency"}
    prob.close()
    return r


def quantiser(bsg, peaks, kind, rows, K, bf16, steps=50, warmup=5, scaled=False):
    """bsg_quantize / bsg_quantize_bf16 on a rows x K activation (float32 or BF16), timed as one
    CUDA-graph replay of `steps` calls.  Algorithmic bytes: the input once, the codes, the
    swizzled scale buffer (and the 4-byte global scale); NVFP4 reads its input twice (tensor
    amax, then the blocks), which the roofline counts as the kernel's own cost, not as bytes."""
    import torch
    from fp4_gemm_blackwell_gb300 import synth
    k = bsg.BSG_MXFP8 if kind == "mxfp8" else bsg.BSG_NVFP4
    x = synth.normal_rowscaled(rows, K, seed=0)
    xd = (torch.from_numpy(synth.as_bf16_bits(x).view(np.int16)) if bf16 else torch.from_numpy(x)).cuda()
    code_bytes = rows * K if kind == "mxfp8" else rows * K // 2
    codes = torch.empty(code_bytes, dtype=torch.uint8, device="cuda")
    sf_bytes = bsg.bsg_sf_bytes(k, rows, K)
    sf = torch.empty(sf_bytes, dtype=torch.uint8, device="cuda")
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    fn = bsg.bsg_quantize_bf16 if bf16 else bsg.bsg_quantize
    if scaled:   # NVFP4 with the global scale given (the tensor's own, from one bsg_quantize call)
        (bsg.bsg_quantize_bf16 if bf16 else bsg.bsg_quantize)(k, xd, rows, K, codes, sf, gs)
        torch.cuda.synchronize()
        fn = lambda k_, x_, r_, K_, c_, s_, g_, st_: bsg.bsg_quantize_nvfp4_scaled(x_, r_, K_, c_, s_, g_, bf16, st_)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn(k, xd, rows, K, codes, sf, gs, stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(steps):
            fn(k, xd, rows, K, codes, sf, gs, stream)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    us = start.elapsed_time(end) * 1e3 / steps
    nbytes = xd.numel() * xd.element_size() + code_bytes + sf_bytes + (4 if kind == "nvfp4" else 0)
    gbs = nbytes / (us * 1e-6) / 1e9
    del g
    return {"us": round(us, 2), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "algorithmic_bytes": nbytes, "input": "bf16" if bf16 else "f32", "shape": [rows, K],
            "launches_per_call": 1 if kind == "mxfp8" or scaled else 3,
            "global_scale": "given" if scaled else ("per tensor (amax pass)" if kind == "nvfp4" else None)}


def launch_loop(bsg, calls=1000):
    """1000 NVFP4 GEMM calls cycling M in {1,16,128,1024} x (N,K) in {(4096,4096),(14336,4096),
    (4096,14336)}, BF16 out: host time per call against device kernel time, (i) one-shot C-ABI
    calls (cached plans) on a stream, (ii) the same 1000 calls captured once in a CUDA graph."""
    shapes = [(m, n, k) for m in (1, 16, 128, 1024) for (n, k) in ((4096, 4096), (14336, 4096), (4096, 14336))]
    ops_a, ops_b = {}, {}
    for (m, n, k) in shapes:
        if (m, k) not in ops_a:
            ops_a[(m, k)] = Operands(bsg, "nvfp4", m, k, 0)
        if (n, k) not in ops_b:
            ops_b[(n, k)] = Operands(bsg, "nvfp4", n, k, 1)
    L = bsg.lib()
    calls_args = []
    keep = []
    for (m, n, k) in shapes:
        a, b = ops_a[(m, k)], ops_b[(n, k)]
        d = torch.empty(m * n, dtype=torch.int16, device="cuda")
        keep.append(d)
        alpha = float(np.float32(np.float32(a.s) * np.float32(b.s)))
        calls_args.append((d.data_ptr(), a.codes.data_ptr(), b.codes.data_ptr(), a.sf.data_ptr(), b.sf.data_ptr(),
                           None, alpha, 0, m, n, k, bsg.BSG_OUT_BF16))
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream

    def issue(i):
        st = L.nvfp4_gemm(*calls_args[i % len(calls_args)], sp)
        if st != 0:
            raise bsg.BsgError(st, bsg.bsg_last_error())

    for i in range(len(shapes) * 3):            # plan-cache misses happen here, untimed
        issue(i)
    torch.cuda.synchronize()
    # (i) stream: host enqueue time, then wall time to completion
    t0 = time.perf_counter()
    for i in range(calls):
        issue(i)
    host_stream = (time.perf_counter() - t0) * 1e6 / calls
    torch.cuda.synchronize()
    wall_stream = (time.perf_counter() - t0) * 1e6 / calls
    # device time of the same 1000 kernels, back to back (graph replay timed with events)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(calls):
            issue(i)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        t1 = time.perf_counter()
        g.replay()
        host_graph = (time.perf_counter() - t1) * 1e6 / calls
        end.record(stream)
    torch.cuda.synchronize()
    kernel_us = start.elapsed_time(end) * 1e3 / calls
    bsg.bsg_cache_clear()
    del g
    native = native_launch_loop()
    return {"calls": calls, "shapes": len(shapes), "kernel_us_per_call": round(kernel_us, 3),
            "c_abi": native,
            "stream": {"host_us_per_call": round(host_stream, 3), "wall_us_per_call": round(wall_stream, 3),
                       "host_over_kernel": round(host_stream / kernel_us, 3)},
            "graph": {"host_us_per_call": round(host_graph, 4), "host_over_kernel": round(host_graph / kernel_us, 4)},
            "note": "host time is the enqueue time through the Python ctypes binding"}


def native_launch_loop():
    """The same loop from a compiled C++ caller (fp4_gemm_blackwell_gb300/bsg_launch_loop, built
    with the library): the host cost of the C ABI itself, without the Python FFI."""
    exe = os.path.join(ROOT, "fp4_gemm_blackwell_gb300", "bsg_launch_loop")
    try:
        r = subprocess.run([exe], stdout=subprocess.PIPE, stderr=subprocess.PIPE, timeout=300)
        return json.loads(r.stdout.decode().strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal: the Python-level loop above still stands
        return {"error": str(e)[:200]}


# ---------------------------------------------------------------- the CPU oracle
def oracle_sample(rows, cols):
    """Operands of a rows x cols block of the headline problem's output, quantised by the CPU
    oracle (setup, untimed): the first `rows` rows of A and `cols` rows of B over the full K, each
    with the NVFP4 tensor scale of its whole 8192 x 8192 matrix (the oracle's own function)."""
    from fp4_gemm_blackwell_gb300 import synth
    from oracle import layout as OL
    from oracle import quantize as OQ
    xa = synth.normal_rowscaled(MH, KH, synth.SEED_A)
    xb = synth.normal_rowscaled(NH, KH, synth.SEED_B)
    sa, sb = OQ.nvfp4_global_scale(xa), OQ.nvfp4_global_scale(xb)
    a, sfa, _ = OQ.quantize_nvfp4(xa[:rows], sa)
    b, sfb, _ = OQ.quantize_nvfp4(xb[:cols], sb)
    _, bias = synth.bias(NH)
    return dict(A=a, B=b, SFA=OL.swizzle(sfa), SFB=OL.swizzle(sfb), rows=rows, cols=cols,
                alpha=np.float32(np.float32(sa) * np.float32(sb)), bias=bias[:cols])


def oracle_block(p):
    """One evaluation of the oracle (table decode, float64 GEMM, bias, SiLU, BF16 rounding) on a
    sample block; returns its FLOPs."""
    from oracle import gemm as OG
    OG.reference(OG.NVFP4, p["A"], p["B"], p["SFA"], p["SFB"], p["rows"], p["cols"], KH, alpha=p["alpha"],
                 bias=p["bias"], silu=True, out=OG.BF16)
    return 2.0 * p["rows"] * p["cols"] * KH


def cpu_baseline(budget_s=10.0):
    """The oracle as it stands on a bounded sample of the headline workload: a 64 x 256 block of
    the 8192^3 output over the full K, repeated until about `budget_s` seconds of CPU work."""
    p = oracle_sample(64, 256)
    reps, flops, t0 = 0, 0.0, time.perf_counter()
    while True:
        flops += oracle_block(p)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    tf = flops / dt / 1e12
    return {"value": round(tf, 6), "unit": "TFLOPS", "cores": os.cpu_count(), "kind": "oracle",
            "sample": "%d evaluations of a 64 x 256 output block of NVFP4 8192^3 (full K = 8192; table decode, "
                      "float64 numpy matmul, bias, SiLU, BF16 rounding) in %.1f s; numpy's BLAS uses all %d host "
                      "threads" % (reps, dt, os.cpu_count())}


def reference_arm(args):
    """--impl reference: the CPU oracle is the reference implementation of this workload.  A step
    is a bounded sample of it: a 32 x 64 block of the 8192^3 output over the full K."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    p = oracle_sample(32, 64)
    for _ in range(args.warmup):
        oracle_block(p)
    flops, t0 = 0.0, time.perf_counter()
    for _ in range(args.steps):
        flops += oracle_block(p)
    dt = time.perf_counter() - t0
    tf = flops / dt / 1e12
    sample = ("per step a 32 x 64 output block of NVFP4 8192^3 (full K, bias + SiLU, BF16) by the float64 "
              "oracle on %d host cores" % os.cpu_count())
    line = {"impl": "reference", "metric": METRIC, "value": round(tf, 6), "unit": "TFLOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": headline_config(),
            "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOPS", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(tf, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


CASES = {
    "nvfp4_m128": ("nvfp4", M1, N1, K1, "bf16", True, True),
    "mxfp8_256": ("mxfp8", 256, 256, 256, "bf16", False, False),
    "mxfp8_8192": ("mxfp8", 8192, 8192, 8192, "bf16", False, False),
    "mxfp8_8192_f16": ("mxfp8", 8192, 8192, 8192, "f16", False, False),
    "nvfp4_8192": ("nvfp4", 8192, 8192, 8192, "bf16", True, True),
    "nvfp4_8000": ("nvfp4", 8000, 8192, 8192, "bf16", True, True),
    "nvfp4_m128_l8": ("nvfp4", M1, N1, K1, "bf16", True, True, 8),  # a batch of 8 entries
}


def case_arm(args):
    """--case NAME: one workload, `steps` plain stream launches of its plan after `warmup`
    (for profiler captures and quick timing); prints one JSON line."""
    if args.case in CUBLAS_CASES:
        return cublas_case(args)
    if args.case in QUANT_CASES:
        return quant_case(args)
    import __graft_entry__
    import fp4_gemm_blackwell_gb300 as bsg
    __graft_entry__.build()
    torch.cuda.set_device(0)
    kind, M, N, K, out, bias, silu, *batch = CASES[args.case]
    prob = Problem(bsg, kind, M, N, K, out=out, bias=bias, silu=silu, copies=1, L=batch[0] if batch else 1)
    us, clk = time_launches(lambda stream: prob.plans[0].run(stream), args.steps, args.warmup)
    prob.plans[0].check_status()
    print(json.dumps({"case": args.case, "variant": prob.variant, "us_per_launch": round(us, 3),
                      "tflops": round(prob.flops() / (us * 1e-6) / 1e12, 2),
                      "gbs": round(prob.algorithmic_bytes() / (us * 1e-6) / 1e9, 1),
                      "clocks": clk}), flush=True)
    prob.close()
    return 0


def time_launches(launch, steps, warmup):
    """`steps` launches of launch(stream) after `warmup`, with the clock sampler running: the
    sampler starts first (its start-up is not in the timed region) and the launches queue
    behind a device-side sleep, so the events measure back-to-back execution.  Returns
    (us per launch, clock record)."""
    stream = torch.cuda.Stream()
    clocks = ClockSampler(0)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            launch(stream)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(2e6))
        start.record(stream)
        for _ in range(steps):
            launch(stream)
        end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    return start.elapsed_time(end) * 1e3 / steps, clk


# cuBLAS's block-scaled GEMM (through torch._scaled_mm) on the shapes of the 8192^3 workloads, for
# a vendor-library figure beside the kernels' (no bias or SiLU: a plain GEMM with BF16 output).
# Random code bytes and scale bytes of one binade; the result is not checked (the GPU tests pin the
# scale layout against the same call).
CUBLAS_CASES = {"cublas_nvfp4_8192": "nvfp4", "cublas_mxfp8_8192": "mxfp8"}


def cublas_case(args):
    torch.cuda.set_device(0)
    kind = CUBLAS_CASES[args.case]
    M = N = K = 8192
    g = torch.Generator(device="cuda").manual_seed(1)

    def operand(rows):
        if kind == "nvfp4":
            codes = torch.randint(0, 256, (rows, K // 2), dtype=torch.uint8, device="cuda", generator=g)
            sf = torch.randint(0x30, 0x40, (rows * (K // 16),), dtype=torch.uint8, device="cuda", generator=g)
            return codes.view(torch.float4_e2m1fn_x2), sf.view(torch.float8_e4m3fn)
        codes = torch.randint(0, 256, (rows, K), dtype=torch.uint8, device="cuda", generator=g)
        codes[(codes & 0x7F) == 0x7F] = 0  # no NaN codes
        sf = torch.randint(120, 134, (rows * (K // 32),), dtype=torch.uint8, device="cuda", generator=g)
        return codes.view(torch.float8_e4m3fn), sf.view(torch.float8_e8m0fnu)

    (a, sa), (b, sb) = operand(M), operand(N)
    us, clk = time_launches(lambda stream: torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb,
                                                             out_dtype=torch.bfloat16),
                            args.steps, args.warmup)
    print(json.dumps({"case": args.case, "library": "cuBLAS via torch._scaled_mm " + torch.__version__,
                      "us_per_launch": round(us, 3), "tflops": round(2.0 * M * N * K / (us * 1e-6) / 1e12, 1),
                      "clocks": clk}), flush=True)
    return 0


# The quantisers on an 8192 x 8192 activation: (kind, BF16 input, global scale given).
QUANT_CASES = {"quantize_mxfp8_f32": ("mxfp8", False, False), "quantize_mxfp8_bf16": ("mxfp8", True, False),
               "quantize_nvfp4_f32": ("nvfp4", False, False), "quantize_nvfp4_bf16": ("nvfp4", True, False),
               "quantize_nvfp4_given_f32": ("nvfp4", False, True),
               "quantize_nvfp4_given_bf16": ("nvfp4", True, True)}


def quant_case(args):
    """--case quantize_*: `steps` quantiser calls replayed as one CUDA graph after `warmup`."""
    import __graft_entry__
    import fp4_gemm_blackwell_gb300 as bsg
    __graft_entry__.build()
    torch.cuda.set_device(0)
    kind, bf16, given = QUANT_CASES[args.case]
    r = quantiser(bsg, load_peaks(), kind, 8192, 8192, bf16, steps=args.steps, warmup=args.warmup, scaled=given)
    print(json.dumps(dict({"case": args.case}, **r)), flush=True)
    return 0


METRIC = "block-scaled GEMM TFLOPS & % tensor peak (MXFP8, NVFP4); host µs/call vs kernel"
WORKLOAD = "nvfp4_gemm M=N=K=8192, bf16 bias + SiLU, bf16 out"


def headline_config():
    """The headline's `config`, the same in both arms."""
    return {"workload": WORKLOAD, "M": MH, "N": NH, "K": KH,
            "l2": "operands and output rotate over 2 copies (420 MB > 129 MB L2)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline only (no other workloads, no CPU baseline)")
    ap.add_argument("--case", choices=sorted(CASES) + sorted(CUBLAS_CASES) + sorted(QUANT_CASES),
                    help="time one workload with plain launches and exit")
    args = ap.parse_args()
    if args.case:
        return case_arm(args)
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        return reference_arm(args)

    import __graft_entry__
    import fp4_gemm_blackwell_gb300 as bsg
    rank, world, local, dist = dist_setup(args.gpus)
    if rank == 0:
        __graft_entry__.build()
    if dist:
        dist.barrier()
    bsg.lib()
    barrier = (lambda: dist.barrier()) if dist else None
    peaks = load_peaks()

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    h = headline(bsg, args.steps, args.warmup, barrier)
    clocks = sampler.stop() if rank == 0 else None
    prob = h["problem"]
    ms_max, value = whole_job(h["ms"], prob.flops(), args.steps, world, dist)
    kernel_us = h["ms"] * 1e3 / args.steps
    achieved = prob.flops() / (kernel_us * 1e-6) / 1e12          # TFLOP/s of the one kernel per step
    peak = tensor_peak(peaks, "nvfp4")
    result = None
    if rank == 0:
        extras = {}
        e2e_r = e2e(bsg, min(200, args.steps))
        if not args.quick:
            extras["nvfp4_m128_n4096_k4096_bias_silu"] = skinny_headline(bsg, peaks)
            extras["mxfp8_256_bf16"] = small_config(bsg, peaks)
            extras["nvfp4_m128_l2_warm"] = l2_warm_config(bsg, peaks)
            extras["mxfp8_8192_bf16"] = big_config(bsg, peaks, "mxfp8", 8192, 8192, 8192, "bf16", False, False)
            extras["mxfp8_8192_f16"] = big_config(bsg, peaks, "mxfp8", 8192, 8192, 8192, "f16", False, False)
            extras["nvfp4_8000x8192x8192_bias_silu_bf16"] = big_config(bsg, peaks, "nvfp4", 8000, 8192, 8192, "bf16",
                                                                       True, True)
            extras["nvfp4_8192_bias_silu_residual_factors_bf16"] = big_config(
                bsg, peaks, "nvfp4", 8192, 8192, 8192, "bf16", True, True, residual=True, factors=True)
            extras["nvfp4_m128_residual_factors"] = skinny_config(bsg, peaks, residual=True, factors=True)
            for L in (2, 8):
                extras["nvfp4_batched_l%d_m128_n4096_k4096" % L] = batched_config(bsg, peaks, L)
            extras["nvfp4_grouped_8x4096x4096_moe"] = grouped_config(bsg, peaks)
            extras["nvfp4_m128_pointer_agnostic"] = remap_config(bsg, peaks)
            extras["nvfp4_m128_nvfp4_out"] = nvfp4_out_config(bsg, peaks, M1, N1, K1, steps=400)
            extras["nvfp4_8192_nvfp4_out"] = nvfp4_out_config(bsg, peaks, 8192, 8192, 8192, steps=20)
            extras["launch_loop_1000"] = launch_loop(bsg)
            for kind in ("mxfp8", "nvfp4"):
                for bf in (False, True):
                    extras["quantize_%s_%s_8192x8192" % (kind, "bf16" if bf else "f32")] = quantiser(
                        bsg, peaks, kind, 8192, 8192, bf)
            for bf in (False, True):
                extras["quantize_nvfp4_given_scale_%s_8192x8192" % ("bf16" if bf else "f32")] = quantiser(
                    bsg, peaks, "nvfp4", 8192, 8192, bf, scaled=True)
        cpu = cpu_baseline() if not args.quick else None
        result = {
            "metric": METRIC, "value": round(value, 4), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e2m1 x e2m1 -> f32 accumulate", "data": "synthetic",
            "config": headline_config(),
            "variant": prob.variant,
            "timing": "CUDA events around one CUDA-graph replay of the K plan launches",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": recorded_traffic("bsg_gemm_pair_kernel<nvfp4>", "nvfp4_8192_bias_silu"),
                         "flops_per_launch": prob.flops(), "algorithmic_bytes_per_launch": prob.algorithmic_bytes(),
                         "kernel_us": round(kernel_us, 3),
                         "peak_source": "%s bf16_tflops %.1f (burst cuBLAS GEMM) x 6, the nominal dense FP4 / BF16 "
                                        "ratio 13.5 / 2.25" % (peaks["source"], peaks["bf16_tflops"])},
            "host_us_per_call": {"plan_run_stream": round(h["host_us_per_run"], 3),
                                 "kernel_us_stream_back_to_back": round(h["stream_kernel_us"], 3)},
            "clocks": clocks, "e2e": e2e_r, "gpu_launches": h["launches"], "cpu_baseline": cpu, "extras": extras,
        }
    prob.close()
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
