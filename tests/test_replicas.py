"""The multi-GPU path of the benchmark is N independent replicas (sequences are
independent; no collective sits on the data path).  Its host logic -- the
slowest replica's time, the whole-job throughput, rank 0 alone printing the
reference arm -- runs here as world-size-2 gloo process groups on the CPU."""
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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        # rank r took (10 + r) ms for its steps and (30 - r) ms end to end
        got = bench.max_over_ranks([10.0 + rank, 30.0 - rank], dist, "cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_replica_sets_the_job_time():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == [11.0, 30.0]


def test_whole_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    # 128 verified positions per step and replica, 2 replicas, 10 steps in 1 ms (the slowest)
    assert bench.job_tokens_per_s(128, 2, 10, 1.0) == pytest.approx(2 * 128 * 10 / 1e-3)
    assert bench.job_tokens_per_s(128, 1, 10, 1.0) * 2 == bench.job_tokens_per_s(128, 2, 10, 1.0)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    bench.run_reference(None, rank=1, world=2)     # returns at once, without work or output
    assert capsys.readouterr().out == ""
