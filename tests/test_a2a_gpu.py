"""The Ulysses all-to-all across GPUs, on one GPU: P ranks emulated in one
process.  Each rank's send buffer comes from the library's pack kernel, the
exchange (block s of rank r's send buffer lands as block r of rank s's
receive buffer) is done with plain device copies, and each rank's result is
checked bit for bit against the oracle's index map; the inverse exchange
restores every sequence shard.  A one-rank NCCL group runs the public
exchange calls themselves (with one rank the collective has nothing to
move, but the pack, the collective and the receive views run on the GPU)."""
import os
import socket

import pytest
import torch

from parity_utils import Guards, bytes_equal

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("P,T,H,d,dtype", [
    (4, 16384, 32, 128, torch.bfloat16),   # Qwen3-4B query heads, N = 65536 over 4 ranks
    (4, 16384, 8, 128, torch.bfloat16),    # its KV heads
    (2, 100, 4, 64, torch.float32),        # ragged: 100 tokens per rank
    (8, 64, 8, 128, torch.bfloat16),       # one head per rank
])
def test_emulated_exchange_bit_exact(uly, oracle_mod, P, T, H, d, dtype):
    g = torch.Generator().manual_seed(P * 1000 + T + H)
    x_seq = torch.randn(P, 1, T, H, d, generator=g).to(dtype)
    ref = oracle_mod.seq_to_head(x_seq, P)                      # [P][1][N][H/P][d]
    xd = x_seq.cuda()
    G = Guards()
    sends = [uly.ulysses_a2a_pack(xd[r], P, out=G.empty((P, 1, T, H // P, d), dtype)) for r in range(P)]
    for r in range(P):
        head = torch.cat([sends[s][r] for s in range(P)], dim=1)   # [1][N][H/P][d], source order
        assert bytes_equal(head, ref[r]), r
    # inverse: rank r sends block s of its head shard to rank s
    heads = [ref[r].cuda().contiguous() for r in range(P)]
    for r in range(P):
        recv = torch.stack([heads[s].view(P, T, H // P, d)[r] for s in range(P)]).unsqueeze(1)
        back = uly.ulysses_a2a_unpack(recv.contiguous(), P, out=G.empty((1, T, H, d), dtype))
        assert bytes_equal(back, x_seq[r]), r
    assert uly.ulysses_get_device_status()[0] == 0
    G.check()


def test_one_rank_nccl_exchange(uly):
    import torch.distributed as dist
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    store = dist.TCPStore("127.0.0.1", port, 1, is_master=True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        x = torch.randn(1, 256, 8, 128, device="cuda").to(torch.bfloat16)
        head = uly.ulysses_all_to_all_seq_to_head(x)
        assert bytes_equal(head, x)                      # one rank holds every head
        back = uly.ulysses_all_to_all_head_to_seq(head)
        assert bytes_equal(back, x)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
