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


def test_committed_tokens_per_s():
    sys.path.insert(0, ROOT)
    import bench
    import numpy as np
    # 4 sequences committing 1 + (3, 0, 2, 1) tokens per step, 10 steps in 2 ms, 2 replicas
    assert bench.committed_tokens_per_s(np.array([3, 0, 2, 1]), 2, 10, 2.0) == pytest.approx(10 * 2 * 10 / 2e-3)
    assert bench.committed_tokens_per_s(None, 1, 10, 2.0) is None
    assert bench.committed_tokens_per_s(torch.tensor([0, 0], dtype=torch.int32).numpy(), 1, 1, 1.0) == \
        pytest.approx(2 / 1e-3)


def test_result_line_carries_the_contract_keys():
    """The benchmark's JSON line, built on the host from a stand-in of the decode step (CPU tensors
    in place of the device ones): every key the contract asks for, and the whole-job value."""
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    import numpy as np
    from lossless_speculative_verification_gb300 import synth

    class FakeStep(bench.DeviceStep):
        def __init__(self):
            self.name, self.w = "decode", synth.WORKLOADS["decode"]
            self.layers = [object()]
            self.T = self.w.dims.T
            self.layer_counts = [torch.ones(self.w.dims.E, dtype=torch.int32)]
            self.logits = object()
            self.alen = torch.tensor([3, 1, 0, 2] * 8, dtype=torch.int32)
            self.launches = 5

    args = argparse.Namespace(steps=20, warmup=5)
    m = dict(total_ms=2.0, layer_ms=0.09, accept_ms=0.016, eager_ms=0.12, e2e_total=6.0, h2d=100, d2h=10,
             clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 7}, one_graph=True)
    line = bench.result_line(args, FakeStep(), m, 1, {"value": 50.0, "unit": "tokens/s", "cores": 1,
                                                      "kind": "oracle", "sample": "x"})
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
                "cpu_baseline", "committed_tokens_per_s"):
        assert key in line, key
    assert line["value"] == pytest.approx(128 * 20 / 2e-3)
    assert line["ms_per_step"] == pytest.approx(0.1)
    assert line["e2e"]["value"] == pytest.approx(128 * 20 / 6e-3)
    assert line["gpu_launches"] == 100
    assert line["committed_tokens_per_s"] == pytest.approx(np.sum(np.array([3, 1, 0, 2] * 8) + 1) * 20 / 2e-3)
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in line["roofline"], key
    assert line["roofline"]["frac"] == pytest.approx(line["roofline"]["achieved"] / line["roofline"]["peak"])
    assert "workload" in line["config"]
