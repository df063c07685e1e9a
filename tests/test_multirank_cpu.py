"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): each
rank owns a disjoint request shard (weak scaling, no data-path collective)
and the whole-job numbers are the slowest rank's time and the sum of the
ranks' tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    reqs = bench.rank_requests(rank, 3)
    ms = [10.0, 25.0][rank]
    ms_e2e = [12.0, 11.0][rank]
    tokens = [224 * 3, 100][rank]
    res = bench.reduce_over_ranks(ms, ms_e2e, tokens, world, torch.device("cpu"))
    gathered = [None] * world
    dist.all_gather_object(gathered, reqs)
    if rank == 0:
        out.put((res, gathered))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_shard_requests_and_reduce_timings():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res, shards = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ms, ms_e2e, tokens = res
    assert ms == 25.0 and ms_e2e == 12.0 and tokens == 224 * 3 + 100
    assert shards == [[0, 1, 2], [3, 4, 5]]
    assert not set(shards[0]) & set(shards[1])


def test_single_rank_reduction_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.0, 4.0, 5, 1, None) == (3.0, 4.0, 5.0)
