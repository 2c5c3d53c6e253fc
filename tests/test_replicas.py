"""Replicas-only multi-GPU plumbing of bench.py, on the CPU with two gloo ranks: the
timed region's barrier, the max-over-ranks step time and the whole-job throughput."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        local_ms = [12.5, 20.0][rank]          # the two ranks' own timed regions
        dist.barrier()
        slowest = bench.max_over_ranks(local_ms, world)
        value = bench.job_throughput_gbs(world, 1_000_000, slowest / 10)  # 10 steps
        out[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_job_throughput():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()  # no fork of this multi-threaded process
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0][0] == out[1][0] == 20.0             # both ranks see the slowest time
    # 2 replicas x 1 MB per step, 2.0 ms per step -> 1.0 GB/s for the whole job
    assert out[0][1] == pytest.approx(1.0)
    assert out[1][1] == pytest.approx(1.0)


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput_gbs(1, 2_000_000_000, 1000.0) == pytest.approx(2.0)
