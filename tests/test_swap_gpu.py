"""GPU parity of the seq<->head swaps: bit-exact against the oracle's index
map, for both dtypes, ragged token chunks, P = 1 and the workload shapes."""
import pytest
import torch

import oracle
from parity_utils import Guards, bytes_equal
from ulysses_inputs import WORKLOADS, draw_seq_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("P,B,N,H,d", [
    (2, 1, 256, 4, 64),      # the fp32 workload's shape
    (4, 1, 8192, 32, 128),   # Qwen3-4B query heads
    (4, 1, 8192, 8, 128),    # Qwen3-4B KV heads
    (4, 2, 1000, 8, 128),    # ragged: 250 tokens per shard, two batches
    (8, 1, 8 * 37, 8, 64),   # one head per rank, odd chunk
    (1, 1, 96, 4, 128),      # P = 1: the swap is the identity
    (4, 3, 4 * 300, 16, 64),
    (2, 1, 8, 400, 128),     # 200 heads per shard: a 100 KB row (fp32) leaves the copy ring one stage
])
def test_swap_bit_exact(uly, oracle_mod, dtype, P, B, N, H, d):
    g = torch.Generator().manual_seed(N + H)
    x = torch.randn(P, B, N // P, H, d, generator=g).to(dtype)
    xd = x.cuda()
    g = Guards()
    h = g.empty((P, B, N, H // P, d), dtype, float("nan"))
    uly.ulysses_seq_to_head(xd, h, P)
    ref = oracle_mod.seq_to_head(x, P)
    assert bytes_equal(h, ref)
    back = g.full_like(xd, float("nan"))
    uly.ulysses_head_to_seq(h, back, P)
    assert bytes_equal(back, x)
    st, site = uly.ulysses_get_device_status()
    assert st == 0, hex(site)
    g.check()


@pytest.mark.parametrize("name", ["qwen3_4b_n65536", "single_shard_n1m"])
def test_swap_full_size(uly, oracle_mod, name):
    """The long-context workloads, swap checked in full against the oracle."""
    w = WORKLOADS[name]
    seq = draw_seq_inputs(w, seed=2, device="cuda", want_dout=False)
    for key, H in (("q", w.Hq), ("k", w.Hkv)):
        x = seq[key]
        h = torch.empty(w.P, w.B, w.N, H // w.P, w.d, dtype=x.dtype, device="cuda")
        uly.ulysses_seq_to_head(x, h, w.P)
        ref = oracle_mod.seq_to_head(x.cpu(), w.P)
        assert bytes_equal(h, ref)
        back = torch.empty_like(x)
        uly.ulysses_head_to_seq(h, back, w.P)
        assert torch.equal(back.view(torch.int16), x.view(torch.int16))
        del h, back, ref
    assert uly.ulysses_get_device_status()[0] == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("P,B,N,Hq,Hkv,d", [
    (4, 1, 8192, 32, 8, 128),   # Q, K, V of the Qwen3-4B shapes
    (4, 2, 1000, 8, 4, 128),    # ragged: 250 tokens per shard, two batches
    (2, 1, 256, 4, 4, 64),      # the fp32 workload's shape
    (8, 1, 8 * 37, 8, 8, 64),   # one head per rank, odd chunk
])
def test_swap_batch_bit_exact(uly, oracle_mod, dtype, P, B, N, Hq, Hkv, d):
    """Q, K, V to the head layout in one launch, then O back while dO comes in
    (two directions in one launch), then dQ, dK, dV back: every tensor equals
    the oracle's index map bit for bit, and nothing is written outside it."""
    g = torch.Generator().manual_seed(N + Hq + Hkv)
    seqs = {n: torch.randn(P, B, N // P, H, d, generator=g).to(dtype)
            for n, H in (("q", Hq), ("k", Hkv), ("v", Hkv), ("dout", Hq))}
    dev = {n: x.cuda() for n, x in seqs.items()}
    G = Guards()
    heads = {n: G.empty((P, B, N, x.shape[3] // P, d), dtype, float("nan")) for n, x in seqs.items()}
    uly.ulysses_swap_batch([(dev[n], heads[n], True) for n in ("q", "k", "v")], P)
    for n in ("q", "k", "v"):
        assert bytes_equal(heads[n], oracle_mod.seq_to_head(seqs[n], P)), n
    # O back (here: the head-layout Q stands in for O) while dO comes in
    o_seq = G.full_like(dev["q"], float("nan"))
    uly.ulysses_swap_batch([(heads["q"], o_seq, False), (dev["dout"], heads["dout"], True)], P)
    assert bytes_equal(o_seq, seqs["q"])
    assert bytes_equal(heads["dout"], oracle_mod.seq_to_head(seqs["dout"], P))
    back = {n: G.full_like(dev[n], float("nan")) for n in ("q", "k", "v")}
    uly.ulysses_swap_batch([(heads[n], back[n], False) for n in ("q", "k", "v")], P)
    for n in ("q", "k", "v"):
        assert bytes_equal(back[n], seqs[n]), n
    st, site = uly.ulysses_get_device_status()
    assert st == 0, hex(site)
    G.check()


def _random_swap_cases(n, seed=99):
    """Seeded random swap shapes: P in 1..8, H a multiple of P (up to 64
    heads), N a multiple of P (ragged token chunks), B in 1..3, d 64 or 128."""
    import numpy as np
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        P = int(rng.choice([1, 2, 3, 4, 8]))
        H = P * int(rng.integers(1, max(2, 64 // P + 1)))
        N = P * int(rng.integers(1, 400))
        out.append((P, int(rng.integers(1, 4)), N, H, int(rng.choice([64, 128]))))
    return out


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("P,B,N,H,d", _random_swap_cases(8))
def test_swap_random_shapes_bit_exact(uly, oracle_mod, dtype, P, B, N, H, d):
    test_swap_bit_exact(uly, oracle_mod, dtype, P, B, N, H, d)
