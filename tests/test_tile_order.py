"""The tile walk order the bf16 attention kernels use (host logic, no GPU).

With packed documents the attention calls sort the 128-row tiles by the
length of their walks, longest first (include/ulysses.h,
ulysses_attn_tile_order).  The walks are recomputed here by brute force over
tokens, from the mask's definition (same document, and j <= i when causal):
a query tile's walk spans the key tiles between the smallest and the largest
key any of its rows may attend to; a key tile's walk spans the query tiles
between the smallest and the largest row that may attend to any of its keys.
"""
import numpy as np
import pytest

from ulysses_inputs import cu_seqlens_from_lengths, doc_lengths


def _doc_of(N, cu):
    if cu is None:
        return np.zeros(N, dtype=np.int64)
    return np.searchsorted(np.asarray(cu[1:-1]), np.arange(N), side="right")


def _walks_brute(N, causal, cu, for_bwd):
    doc = _doc_of(N, cu)
    n = (N + 127) // 128
    walks = np.zeros(n, dtype=np.int64)
    idx = np.arange(N)
    for t in range(n):
        lo_tok, hi_tok = 128 * t, min(128 * t + 128, N)
        tiles = set()
        for x in range(lo_tok, hi_tok):
            same = doc == doc[x]
            if for_bwd:  # rows i that may attend to key x
                ok = same & (idx >= x) if causal else same
            else:        # keys j that row x may attend to
                ok = same & (idx <= x) if causal else same
            sel = idx[ok]
            tiles.add(int(sel.min()) // 128)
            tiles.add(int(sel.max()) // 128)
        walks[t] = max(tiles) - min(tiles) + 1
    return walks


@pytest.fixture(scope="module")
def uly():
    import long_context_sequence_head_gb300 as m
    m.load(build_if_missing=True)
    return m


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("for_bwd", [False, True])
def test_without_documents_is_index_order(uly, causal, for_bwd):
    N = 1000  # 8 tiles, ragged tail
    order = uly.ulysses_attn_tile_order(N, causal, None, for_bwd)
    n = (N + 127) // 128
    expect = np.arange(n) if for_bwd else np.arange(n)[::-1]
    assert np.array_equal(order, expect), order


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("for_bwd", [False, True])
@pytest.mark.parametrize("case", ["one-token docs", "straddling", "zero-length docs", "recipe"])
def test_documents_longest_walk_first(uly, causal, for_bwd, case):
    if case == "one-token docs":
        N, cu = 700, [0, 100, 101, 350, 700]
    elif case == "straddling":
        N, cu = 1500, [0, 129, 300, 301, 1100, 1500]
    elif case == "zero-length docs":
        N, cu = 900, [0, 0, 128, 128, 300, 900, 900]
    else:
        N = 4096
        cu = list(cu_seqlens_from_lengths(doc_lengths(N, 4, seed=5, lo=64, hi=900)))
    order = uly.ulysses_attn_tile_order(N, causal, cu, for_bwd)
    n = (N + 127) // 128
    assert sorted(order.tolist()) == list(range(n))  # a permutation
    walks = _walks_brute(N, causal, cu, for_bwd)
    w = walks[order]
    assert np.all(w[:-1] >= w[1:]), (order, w)      # longest first
    # ties keep the plain order: later tiles first forward, earlier backward
    for a, b in zip(order[:-1], order[1:]):
        if walks[a] == walks[b]:
            assert (a < b) if for_bwd else (a > b), (a, b)


def test_order_changes_with_documents(uly):
    """The order is not the index order once documents are packed (the
    reason the attention calls sort at all)."""
    N = 4096
    cu = list(cu_seqlens_from_lengths(doc_lengths(N, 4, seed=5, lo=64, hi=900)))
    assert not np.array_equal(uly.ulysses_attn_tile_order(N, True, cu, True), np.arange(32))


@pytest.mark.parametrize("args", [
    dict(N=0, causal=True, cu_seqlens=None),
    dict(N=256, causal=True, cu_seqlens=[0, 100, 200]),      # does not end at N
    dict(N=256, causal=True, cu_seqlens=[0, 200, 100, 256]),  # decreasing
    dict(N=256, causal=True, cu_seqlens=[5, 256]),            # does not start at 0
])
def test_rejects_what_the_attention_calls_reject(uly, args):
    with pytest.raises(uly.UlyssesError):
        uly.ulysses_attn_tile_order(args["N"], args["causal"], args["cu_seqlens"], False)
