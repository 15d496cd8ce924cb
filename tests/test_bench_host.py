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
