"""The multi-rank path of bench.py (replicas, one per GPU, no data-path
collective) on CPU: two gloo ranks over 127.0.0.1 agree on the slowest
rank's time, and the whole-job throughput counts every rank's bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        dist.barrier()
        ms = bench.max_over_ranks(1.0 + 2.5 * rank, world, torch.device("cpu"))
        out[rank] = ms
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork of this threaded process
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == pytest.approx(3.5)


def test_whole_job_throughput_counts_every_rank():
    one = bench.whole_job_gbps(10 ** 9, 1.0, 1)
    assert one == pytest.approx(1000.0)
    assert bench.whole_job_gbps(10 ** 9, 1.0, 4) == pytest.approx(4 * one)
    assert bench.max_over_ranks(2.0, 1, torch.device("cpu")) == 2.0


def test_reference_arm_runs_on_rank_0_only():
    # under torchrun with two ranks the other rank exits 0 without work or output
    import subprocess
    import sys
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl",
                        "reference", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
