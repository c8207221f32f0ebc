"""The bench's N-rank bookkeeping on CPU (gloo, world_size 2): every rank
gets the slowest rank's times, and the job throughput counts the units of
all ranks over that time (weak scaling, sequences sharded by rank)."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        got = bench.slowest_rank([1.0 + rank, 5.0 - rank], "cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_gloo_two_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == [2.0, 5.0] and out[1] == [2.0, 5.0]


def test_job_rate_counts_all_ranks():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_rate(1e9, 1, 10.0)
    assert abs(one - 100.0) < 1e-9
    assert abs(bench.job_rate(1e9, 4, 10.0) - 4 * one) < 1e-9
    assert bench.slowest_rank([3.0, 1.5], "cpu") == [3.0, 1.5]   # single process
