"""Host logic of the multi-process bench path, on CPU with gloo (world size 2):
each rank runs its own requests; the job's time is the max over ranks and its
tokens the sum."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (rank, world, rank)
    secs, toks = bench.aggregate(0.5 + rank, 32 * (rank + 1), world)
    bench.barrier(world)
    q.put((rank, secs, toks))
    dist.destroy_process_group()


def test_aggregate_max_time_sum_tokens_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 1.5, 96), (1, 1.5, 96)]


def test_aggregate_single_rank_is_identity():
    import bench
    assert bench.aggregate(2.0, 7, 1) == (2.0, 7)
