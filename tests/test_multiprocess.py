"""The multi-GPU path of the benchmark on the CPU: two gloo ranks (world size 2,
127.0.0.1).  The paged KV cache partitions by sequence with no exchange step,
so each rank runs its own replica batch; the host logic is the max over ranks
of the step time and the whole-job (weak-scaling) throughput."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = [10.0 + rank, 3.0 * (world - rank)]          # each rank's own timings (ms)
    out[rank] = bench.max_over_ranks(times, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == out[1] == [11.0, 6.0]


def test_weak_scaling_value_counts_every_rank():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    one = bench.weak_scaling_value(543_000_000, 1, 0.1)
    assert one == pytest.approx(5430.0)
    assert bench.weak_scaling_value(543_000_000, 4, 0.1) == pytest.approx(4 * one)
    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]   # no process group: identity
