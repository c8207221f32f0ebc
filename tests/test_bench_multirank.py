"""The bench's N-rank path on CPU (gloo, world_size 2): the ranks' shards of
one workload cover every sequence of the job's batch exactly once, with the
batch's lengths; every rank gets the slowest rank's times; the job
throughput counts the units of all ranks over that time (weak scaling)."""
import os
import socket
import sys

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORKLOADS = ("tiny", "llama8b", "ragged", "longctx", "gemma_write", "prefill", "prefill_hd256")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    from quantized_paged_kv_reshape_gb300 import workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        out[("slowest", rank)] = bench.slowest_rank([1.0 + rank, 5.0 - rank], "cpu")
        for name in WORKLOADS:
            w = W.rank_workload(name, world, rank)
            mine = [(int(g), int(n)) for g, n in zip(w.notes["global_seqs"], w.seq_lens)]
            got = [None] * world
            dist.all_gather_object(got, mine)
            out[(name, rank)] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_ranks_partition_one_workload_gloo_two_ranks():
    sys.path.insert(0, ROOT)
    from quantized_paged_kv_reshape_gb300 import workloads as W
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[("slowest", 0)] == [2.0, 5.0] and out[("slowest", 1)] == [2.0, 5.0]
    for name in WORKLOADS:
        lens = W.global_lengths(name, world)
        assert lens.size == world * W.make(name).num_seqs
        views = [out[(name, r)] for r in range(world)]
        assert views[0] == views[1]                       # every rank sees the same split
        owned = [g for shard in views[0] for g, _ in shard]
        assert sorted(owned) == list(range(lens.size))    # each sequence exactly once
        for shard in views[0]:
            for g, n in shard:
                assert n == lens[g]
        sizes = [len(shard) for shard in views[0]]
        assert max(sizes) - min(sizes) <= 1


def test_one_rank_is_the_workload_itself():
    sys.path.insert(0, ROOT)
    from quantized_paged_kv_reshape_gb300 import workloads as W
    for name in WORKLOADS:
        w, base = W.rank_workload(name, 1, 0), W.make(name)
        assert np.array_equal(w.seq_lens, base.seq_lens)
        assert np.array_equal(w.notes["global_seqs"], np.arange(base.num_seqs))


def test_shard_sequences_rejects_bad_rank():
    sys.path.insert(0, ROOT)
    from quantized_paged_kv_reshape_gb300 import workloads as W
    import pytest
    with pytest.raises(ValueError):
        W.shard_sequences(8, 2, 2)


def test_job_rate_counts_all_ranks():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_rate(1e9, 1, 10.0)
    assert abs(one - 100.0) < 1e-9
    assert abs(bench.job_rate(1e9, 4, 10.0) - 4 * one) < 1e-9
    assert bench.slowest_rank([3.0, 1.5], "cpu") == [3.0, 1.5]   # single process
