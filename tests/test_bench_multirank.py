"""The benchmark's multi-rank host logic on two gloo ranks (CPU): the job time
is the slowest rank's, the job rate sums the replicas, and only rank 0 runs the
reference arm."""
import os
import socket
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        rate = bench.job_rate(1000, world, ms)
        line = bench.run_reference(types.SimpleNamespace(warmup=0, steps=1, cpu_seconds=0.0), rank, world) \
            if rank != 0 else "rank0"
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{ms} {rate} {line}")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_replicas(tmp_path):
    world, port = 2, _free_port()
    times = [12.5, 20.0]
    mp.start_processes(_rank_main, args=(world, port, times, str(tmp_path)), nprocs=world, start_method="spawn")
    for r in range(world):
        ms, rate, line = open(tmp_path / f"r{r}.txt").read().split(" ", 2)
        assert float(ms) == 20.0                        # every rank reports the slowest rank's time
        assert float(rate) == pytest.approx(2 * 1000 / 0.020)
        assert line == ("rank0" if r == 0 else "None")  # other ranks skip the reference arm


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    assert bench.job_rate(10, 1, 2.0) == pytest.approx(5000.0)
