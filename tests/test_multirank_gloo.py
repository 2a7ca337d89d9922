"""The N>1 benchmark path on CPU: two gloo ranks run the bench's barrier +
max-over-ranks timing logic and its whole-job throughput (replicas, weak
scaling).  No GPU: the ranks' 'times' are made up on the host, one of them
slower, and one rank leaves between steps to check the survivor learns of it
through the store rather than hanging."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    my_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    ms = bench.max_over_ranks(my_ms, dist)
    tput = bench.whole_job_throughput(world, 2.0e12, ms)
    q.put((rank, ms, tput))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tput in res:
        assert ms == 15.0                           # the slowest rank decides
        assert tput == pytest.approx(2 * 2.0e12 / 15e-3 / 1e12)


def _leaver(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    store = dist.TCPStore("127.0.0.1", port + 1, world, is_master=(rank == 0), timeout=__import__("datetime").timedelta(seconds=30))
    dist.init_process_group("gloo", rank=rank, world_size=world, store=dist.PrefixStore("pg", store))
    dist.barrier()
    if rank == 1:
        # leave between steps: announce it on the host, no collective in flight
        store.set("rank1_left", "1")
        q.put((rank, "left"))
        return
    # rank 0 checks the store before its next launch instead of entering a
    # collective the other rank will never join
    store.wait(["rank1_left"])
    q.put((rank, store.get("rank1_left").decode()))


def test_rank_leaving_between_steps_is_seen_on_the_host():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_leaver, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    assert res == {0: "1", 1: "left"}
