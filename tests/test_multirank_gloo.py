"""The N>1 benchmark path on CPU: two gloo ranks run the bench's barrier +
max-over-ranks timing logic and its whole-job throughput (replicas, weak
scaling).  No GPU: the ranks' 'times' are made up on the host, one of them
slower, and one rank leaves between steps to check the survivor learns of it
through the store rather than hanging.  The Ulysses all-to-all across ranks
(the exchange a multi-GPU run makes) runs on 2 and 4 gloo ranks."""
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


def _a2a_worker(rank, world, port, q):
    """One rank of the Ulysses all-to-all on CPU: the local pack/unpack steps
    are the oracle's index maps here (the library's kernels need a GPU); the
    exchange, the block order and the buffer views are the product's."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch
    import oracle
    import long_context_sequence_head_gb300 as uly

    def seq_to_head(x_seq, x_head, P, stream=None):
        x_head.copy_(oracle.seq_to_head(x_seq, P))
        return x_head

    def head_to_seq(x_head, x_seq, P, stream=None):
        x_seq.copy_(oracle.head_to_seq(x_head, P))
        return x_seq
    uly.ulysses_seq_to_head = seq_to_head
    uly.ulysses_head_to_seq = head_to_seq
    P = world
    out = []
    for T, H, d, dt in ((4 * P, 4 * P, 8, torch.bfloat16), (2 * P, 2 * P, 16, torch.float32)):
        g = torch.Generator().manual_seed(100 + T + H)
        x_seq = torch.randn(P, 1, T, H, d, generator=g).to(dt)   # every rank draws the same global tensor
        mine = x_seq[rank].clone()                               # [1][T][H][d]: tokens [rank*T, (rank+1)*T)
        head = uly.ulysses_all_to_all_seq_to_head(mine)
        ref = oracle.seq_to_head(x_seq, P)[rank]                 # [1][N][H/P][d]: heads of block `rank`
        ok_fwd = head.shape == ref.shape and torch.equal(head.view(torch.uint8), ref.contiguous().view(torch.uint8))
        back = uly.ulysses_all_to_all_head_to_seq(head)
        ok_back = torch.equal(back.view(torch.uint8), mine.view(torch.uint8))
        out.append((ok_fwd, ok_back))
    try:
        uly.ulysses_a2a_pack(torch.zeros(1, P + 1, P, 8), P)     # T % P != 0 is refused
        refused = False
    except ValueError:
        refused = True
    q.put((rank, out, refused))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_all_to_all_exchange_matches_the_index_map(world):
    """Each gloo rank holds one sequence shard; after the exchange it holds the
    oracle's head shard bit for bit, and the inverse exchange restores its
    sequence shard."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_a2a_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, cases, refused in res:
        assert refused, rank
        for ok_fwd, ok_back in cases:
            assert ok_fwd and ok_back, (rank, cases)
