"""Pins for the oracle's seq<->head swap (CPU only).

The swap is pinned to
* the Ulysses all-to-all diagram (golden fixture ``ulysses_p2_diagram.txt``),
* an independent statement of the permutation with torch view/permute,
* the two round trips being the identity, bit for bit, for several dtypes.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_diagram():
    spec = {"before": {}, "after": {}}
    with open(os.path.join(GOLDEN, "ulysses_p2_diagram.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] in ("N", "H", "P"):
                spec[parts[0]] = int(parts[1])
            else:
                kind, rank = parts[0], int(parts[1])
                spec[kind][rank] = dict(tokens=(int(parts[3]), int(parts[4])),
                                        heads=(int(parts[6]), int(parts[7])))
    return spec


def _tagged_seq(P, B, N, H, d):
    """Element value encodes (batch, global token, head, k) uniquely (int64)."""
    Np = N // P
    x = torch.empty(P, B, Np, H, d, dtype=torch.int64)
    for s in range(P):
        for b in range(B):
            for t in range(Np):
                n = s * Np + t
                for h in range(H):
                    for k in range(d):
                        x[s, b, t, h, k] = ((b * N + n) * H + h) * d + k
    return x


def test_diagram_p2(oracle_mod):
    """Rank r after the swap holds every token, in order, for head block r."""
    spec = _read_diagram()
    N, H, P = spec["N"], spec["H"], spec["P"]
    d, B = 3, 1
    x = _tagged_seq(P, B, N, H, d)
    # the 'before' rows of the diagram describe the seq layout itself
    Np = N // P
    for r, rng in spec["before"].items():
        assert rng["tokens"] == (r * Np, (r + 1) * Np) and rng["heads"] == (0, H)
    y = oracle_mod.seq_to_head(x, P)
    assert y.shape == (P, B, N, H // P, d)
    for r, rng in spec["after"].items():
        t0, t1 = rng["tokens"]
        h0, h1 = rng["heads"]
        assert (t1 - t0) == N and (h1 - h0) == H // P
        for n in range(N):
            for hh in range(H // P):
                for k in range(d):
                    tag = int(y[r, 0, n, hh, k])
                    assert tag % d == k
                    head = (tag // d) % H
                    tok = (tag // (d * H)) % N
                    assert tok == t0 + n
                    assert head == h0 + hh
    # the second all-to-all returns to the 'before' layout
    z = oracle_mod.head_to_seq(y, P)
    assert torch.equal(z, x)


def _torch_statement_seq_to_head(x, P):
    # x [P][B][N/P][H][d] -> split heads into (P, H/P), move the head block
    # axis to the front, then merge (source rank, local token) into tokens.
    Ps, B, Np, H, d = x.shape
    y = x.reshape(Ps, B, Np, P, H // P, d).permute(3, 1, 0, 2, 4, 5)
    return y.reshape(P, B, Ps * Np, H // P, d).contiguous()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float64, torch.int16])
@pytest.mark.parametrize("P,B,N,H,d", [(2, 1, 8, 4, 4), (4, 2, 12, 8, 3), (8, 1, 16, 8, 2),
                                       (1, 1, 5, 3, 2), (4, 3, 8, 4, 16)])
def test_matches_torch_permute(oracle_mod, dtype, P, B, N, H, d):
    g = torch.Generator().manual_seed(P * 1000 + N)
    x = (torch.randn(P, B, N // P, H, d, generator=g) * 100).to(dtype)
    y = oracle_mod.seq_to_head(x, P)
    ref = _torch_statement_seq_to_head(x, P)
    assert torch.equal(y.view(torch.uint8) if dtype != torch.float64 else y, ref.view(torch.uint8)
                       if dtype != torch.float64 else ref)
    # round trips, bit for bit
    back = oracle_mod.head_to_seq(y, P)
    assert torch.equal(back.contiguous().view(torch.uint8), x.contiguous().view(torch.uint8))
    yy = oracle_mod.seq_to_head(oracle_mod.head_to_seq(ref, P), P)
    assert torch.equal(yy.view(torch.uint8), ref.view(torch.uint8))


def test_swap_is_a_permutation(oracle_mod):
    """Every element lands exactly once (no duplicated or dropped element)."""
    P, B, N, H, d = 4, 2, 16, 8, 2
    x = _tagged_seq(P, B, N, H, d)
    y = oracle_mod.seq_to_head(x, P)
    a = np.sort(x.numpy().ravel())
    b = np.sort(y.numpy().ravel())
    assert np.array_equal(a, b)
    assert len(np.unique(b)) == b.size
