"""Multi-rank host logic of bench.py, on CPU with two gloo ranks.

The decode path shards into independent replicas (no data exchange); what
runs across ranks is the timing reduction: the job's time is the slowest
rank's, and the throughput counts every rank's tokens.
"""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, local = bench.dist_env()
    mine = 1.0 + rank                     # rank 1 is the slow one
    slowest = bench.max_over_ranks(mine, w)
    tput = bench.job_throughput(tokens_per_step=4, steps=10, world=w, seconds=slowest)
    dist.barrier()
    q.put((r, local, w, slowest, tput))
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r, local, w, slowest, tput) in enumerate(got):
        assert (r, local, w) == (rank, rank, 2)
        assert slowest == 2.0                         # max over ranks
        assert tput == pytest.approx(2 * 4 * 10 / 2.0)  # all ranks' tokens over the slowest time


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1, 50, 1, 0.5) == 100.0
