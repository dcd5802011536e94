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


def _shard_worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synth
    base, count = bench.rank_requests(32, world, rank)
    w = synth.WORKLOADS["1b-bf16"].with_(batch=count, request_base=base)
    mine = torch.tensor([base, count, float(synth.keys(w, 0, 0, 0, 4).astype(float).sum())],
                        dtype=torch.float64)
    got = [torch.zeros(3, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(got, mine)
    q.put((rank, [tuple(t.tolist()) for t in got]))
    dist.destroy_process_group()


def test_ranks_run_disjoint_requests_gloo():
    # each rank's requests: disjoint ranges covering the job, and different data
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res[0] == res[1]
    ranges = sorted((int(b), int(c)) for b, c, _ in res[0])
    assert ranges == [(0, 32), (32, 32)]
    assert res[0][0][2] != res[0][1][2]


def test_rank_requests_limits():
    import bench
    assert bench.rank_requests(32, 8, 7) == (224, 32)
    with pytest.raises(ValueError):
        bench.rank_requests(300, 8, 0)


def test_aggregate_single_rank_is_identity():
    import bench
    assert bench.aggregate(2.0, 7, 1) == (2.0, 7)
