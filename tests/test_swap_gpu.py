"""GPU parity of the seq<->head swaps: bit-exact against the oracle's index
map, for both dtypes, ragged token chunks, P = 1 and the workload shapes."""
import pytest
import torch

import oracle
from parity_utils import bytes_equal
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
    h = torch.full((P, B, N, H // P, d), float("nan"), dtype=dtype, device="cuda")
    uly.ulysses_seq_to_head(xd, h, P)
    ref = oracle_mod.seq_to_head(x, P)
    assert bytes_equal(h, ref)
    back = torch.full_like(xd, float("nan"))
    uly.ulysses_head_to_seq(h, back, P)
    assert bytes_equal(back, x)
    st, site = uly.ulysses_get_device_status()
    assert st == 0, hex(site)


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
