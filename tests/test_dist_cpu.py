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


def test_host_store_report_deltas():
    import bench
    st = {"host_store_kind": 2, "host_store_pinned": 1}
    created = {"thp_split_page": 3, "pgmigrate_success": 10}
    t0 = {"thp_split_page": 3, "pgmigrate_success": 14}
    t1 = {"thp_split_page": 5, "pgmigrate_success": 14, "thp_split_page_failed": 2}
    r = bench.host_store_report(st, 8704 * 1024, 5632 * 1024, 8704 * 1024, created, t0, t1)
    assert r["layout"] == "transparent huge pages" and r["long_term_pins"] is True
    assert (r["huge_pages_mb"], r["huge_pages_mb_after_timed"], r["pinned_mb"]) == (8704, 5632, 8704)
    # only the counters that moved, over the setup and over the timed steps
    assert r["vm_events"] == {"setup": {"pgmigrate_success": 4},
                              "timed": {"thp_split_page": 2, "thp_split_page_failed": 2}}
    r = bench.host_store_report({"host_store_kind": 0, "host_store_pinned": 0},
                                None, None, None, None, t0, t1)
    assert r["layout"] == "cudaHostAlloc" and r["vm_events"] is None
    assert r["huge_pages_mb"] is None and r["pinned_mb"] is None


def test_proc_readers_on_this_host():
    import bench
    ev = bench.vm_events()
    if ev is not None:  # Linux: the named counters that this kernel has, as integers
        assert set(ev) <= set(bench.VM_EVENTS)
        assert all(isinstance(v, int) and v >= 0 for v in ev.values())
    for kb in (bench.anon_huge_kb(), bench.pinned_kb()):
        assert kb is None or (isinstance(kb, int) and kb >= 0)
