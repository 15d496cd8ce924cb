"""Host logic of bench.py without a GPU: the whole-job aggregation over ranks (two gloo ranks on
CPU, each timing a different region), and the reference arm's rank rule (ranks other than 0 exit
without work)."""

import argparse
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]
        out[rank] = bench.whole_job(ms, 1e12, 10, world, dist, device="cpu")
    finally:
        dist.destroy_process_group()


def test_whole_job_takes_the_slowest_rank_and_counts_every_rank():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    # both ranks see the maximum (5 ms) and 2 ranks x 10 steps x 1 TFLOP over it
    for r in range(world):
        ms, value = res[r]
        assert ms == 5.0
        assert value == pytest.approx(1e12 * 10 * 2 / 5e-3 / 1e12)


def test_whole_job_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job(4.0, 2e9, 100, 1) == (4.0, pytest.approx(2e9 * 100 / 4e-3 / 1e12))


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    assert bench.reference_arm(argparse.Namespace(steps=1, warmup=3, gpus=2)) == 0


def test_algorithmic_bytes_of_the_measured_configurations():
    # the per-launch byte counts the rooflines divide by, against the sums spelled out term by
    # term: codes of A and B, their padded scales, the bias and the 16-bit output
    sys.path.insert(0, ROOT)
    import bench
    # NVFP4 128 x 4096 x 4096 + bias: 262,144 + 32,768 + 8,388,608 + 1,048,576 + 8,192 + 1,048,576
    assert bench.algorithmic_bytes("nvfp4", 128, 4096, 4096, bias=True) == 10_788_864
    # MXFP8 256^3: 65,536 + 2,048 + 65,536 + 2,048 + 131,072
    assert bench.algorithmic_bytes("mxfp8", 256, 256, 256) == 266_240
    # MXFP8 8192^3: two 64 MiB code matrices, two 2 MiB scale buffers, a 128 MiB output
    assert bench.algorithmic_bytes("mxfp8", 8192, 8192, 8192) == 2 * 67_108_864 + 2 * 2_097_152 + 134_217_728
    # NVFP4 8192^3 + bias
    assert bench.algorithmic_bytes("nvfp4", 8192, 8192, 8192, bias=True) == \
        2 * 33_554_432 + 2 * 4_194_304 + 16_384 + 134_217_728
    # ragged M: A's scales padded to 8064 rows
    assert bench.algorithmic_bytes("nvfp4", 8000, 8192, 8192) == \
        8000 * 4096 + 8192 * 4096 + 8064 * 512 + 8192 * 512 + 8000 * 8192 * 2
    # residual and factors; L entries
    base = bench.algorithmic_bytes("nvfp4", 128, 4096, 4096, bias=True)
    assert bench.algorithmic_bytes("nvfp4", 128, 4096, 4096, bias=True, residual=True, factors=True) == \
        base + 128 * 4096 * 2 + (128 + 4096) * 4
    assert bench.algorithmic_bytes("nvfp4", 128, 4096, 4096, bias=True, L=8) == 8 * (base - 8192) + 8192


def test_kernel_source_hash_ignores_comments_only():
    # The traffic records in profiles/traffic.json are keyed by this hash: a comment edit keeps
    # them, any code edit drops them.
    sys.path.insert(0, ROOT)
    import bench
    code = "int f(int x) {  // one\n  /* two\n     lines */ return x + 1;\n}\n"
    assert bench.strip_comments(code) == "int f(int x) {\n   return x + 1;\n}"
    assert bench.strip_comments(code.replace("// one", "// changed")) == bench.strip_comments(code)
    assert bench.strip_comments(code.replace("x + 1", "x + 2")) != bench.strip_comments(code)
    assert bench.recorded_traffic("bsg_gemm_pair_kernel<nvfp4>", "nvfp4_8192_bias_silu") is not None
