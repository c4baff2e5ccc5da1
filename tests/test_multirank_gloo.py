"""The multi-rank path of bench.py on CPU: two gloo ranks, slowest rank's time
and all ranks' tokens (weak scaling, one independent problem per rank)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms, value = bench.aggregate_over_ranks(10.0 + 5.0 * rank, 32768, dist, "cpu")
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork of a process that may hold threads
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    for r in range(world):
        ms, value = out[r]
        assert ms == 15.0  # max over ranks
        assert abs(value - world * 32768 / 0.015) < 1e-6


def test_single_process_aggregation():
    ms, value = __import__("bench").aggregate_over_ranks(20.0, 1000)
    assert ms == 20.0 and abs(value - 50000.0) < 1e-9
