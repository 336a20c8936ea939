"""The N > 1 path of bench.py (replicas: max over ranks of the timed region,
whole-job steps/s) on two gloo ranks on the CPU."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (world, rank, rank)
    seconds = 1.0 + rank  # rank 1 is the slower one
    slowest = bench.max_over_ranks(seconds, world)
    bench.barrier(world)
    out[rank] = (slowest, bench.aggregate(10, slowest, world))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    for r in range(world):
        slowest, value = out[r]
        assert slowest == 2.0
        assert value == 2 * 10 / 2.0
