"""Pins for the oracle's attention forward (CPU only).

* torch fp64 ``scaled_dot_product_attention`` with an explicit boolean mask
  and repeated KV heads (a library routine, independent of the oracle's loops);
* closed forms: N=1, K=0 (uniform weights), one-hot V (softmax rows sum to 1);
* shift invariance of softmax in the keys;
* Ulysses-sharded attention equals unsharded attention;
* packed documents equal attention run on every document separately;
* sampled rows equal the full forward.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F


def _randn(shape, seed, dtype=torch.float64):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64).to(dtype)


def _mask(N, causal, cu):
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    m = torch.ones(N, N, dtype=torch.bool)
    if causal:
        m &= j <= i
    if cu is not None:
        lengths = torch.tensor(np.diff(np.asarray(cu)), dtype=torch.int64)
        doc = torch.repeat_interleave(torch.arange(len(lengths)), lengths)
        m &= doc[:, None] == doc[None, :]
    return m


def _torch_reference(q, k, v, causal, cu, scale):
    # q [S][B][N][Hq][d] -> per (S, B): [Hq][N][d]
    S, B, N, Hq, d = q.shape
    Hkv = k.shape[3]
    G = Hq // Hkv
    mask = _mask(N, causal, cu)
    o = torch.empty_like(q)
    lse = torch.empty(S, B, Hq, N, dtype=torch.float64)
    for s in range(S):
        for b in range(B):
            qq = q[s, b].permute(1, 0, 2)
            kk = k[s, b].permute(1, 0, 2).repeat_interleave(G, dim=0)
            vv = v[s, b].permute(1, 0, 2).repeat_interleave(G, dim=0)
            o[s, b] = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask,
                                                     scale=scale).permute(1, 0, 2)
            scores = torch.einsum("hid,hjd->hij", qq, kk) * scale
            lse[s, b] = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
    return o, lse


CASES = [
    # S, B, N, Hq, Hkv, d, causal, cu
    (1, 1, 7, 2, 2, 4, True, None),
    (2, 2, 13, 4, 2, 8, True, None),
    (1, 1, 16, 4, 1, 8, False, None),
    (2, 1, 20, 2, 1, 4, True, [0, 5, 6, 14, 20]),
    (1, 2, 11, 3, 3, 5, False, [0, 4, 11]),
    (1, 1, 14, 2, 1, 4, True, [0, 0, 5, 5, 9, 14, 14]),  # zero-length documents: first, middle, last
]


@pytest.mark.parametrize("S,B,N,Hq,Hkv,d,causal,cu", CASES)
def test_matches_torch_sdpa(oracle_mod, S, B, N, Hq, Hkv, d, causal, cu):
    q = _randn((S, B, N, Hq, d), 1)
    k = _randn((S, B, N, Hkv, d), 2)
    v = _randn((S, B, N, Hkv, d), 3)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle_mod.attn_fwd(q, k, v, causal=causal, cu_seqlens=cu)
    o_ref, lse_ref = _torch_reference(q, k, v, causal, cu, scale)
    np.testing.assert_allclose(o, o_ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref.numpy(), rtol=1e-12, atol=1e-12)


def test_single_token(oracle_mod):
    q = _randn((1, 1, 1, 2, 8), 4)
    k = _randn((1, 1, 1, 1, 8), 5)
    v = _randn((1, 1, 1, 1, 8), 6)
    o, lse = oracle_mod.attn_fwd(q, k, v, causal=True, scale=0.25)
    for h in range(2):
        np.testing.assert_array_equal(o[0, 0, 0, h], v[0, 0, 0, 0].numpy())
        assert lse[0, 0, h, 0] == pytest.approx(0.25 * float(q[0, 0, 0, h] @ k[0, 0, 0, 0]), abs=1e-15)


@pytest.mark.parametrize("causal,cu", [(True, None), (False, None), (True, [0, 3, 9, 12])])
def test_zero_keys_uniform(oracle_mod, causal, cu):
    """K = 0 makes every allowed score 0: o_i is the mean of the allowed v_j."""
    N, d = 12, 4
    q = _randn((1, 1, N, 2, d), 7)
    k = torch.zeros(1, 1, N, 1, d, dtype=torch.float64)
    v = _randn((1, 1, N, 1, d), 8)
    o, lse = oracle_mod.attn_fwd(q, k, v, causal=causal, cu_seqlens=cu)
    m = _mask(N, causal, cu)
    for h in range(2):
        for i in range(N):
            allowed = m[i].nonzero().flatten()
            np.testing.assert_allclose(o[0, 0, i, h], v[0, 0, allowed, 0].mean(0).numpy(),
                                       rtol=1e-13, atol=1e-14)
            assert lse[0, 0, h, i] == pytest.approx(math.log(len(allowed)), abs=1e-13)


@pytest.mark.parametrize("causal,cu", [(True, None), (False, [0, 6, 10])])
def test_onehot_values_rows_sum_to_one(oracle_mod, causal, cu):
    """V = identity exposes the probabilities: rows sum to 1, zero where masked."""
    N = 10
    q = _randn((1, 1, N, 1, N), 9)
    k = _randn((1, 1, N, 1, N), 10)
    v = torch.eye(N, dtype=torch.float64).reshape(1, 1, N, 1, N)
    o, _ = oracle_mod.attn_fwd(q, k, v, causal=causal, cu_seqlens=cu)
    P = o[0, 0, :, 0, :]
    assert np.all(np.abs(P.sum(1) - 1.0) <= 1e-12)
    m = _mask(N, causal, cu).numpy()
    assert np.all(P[~m] == 0.0)
    assert np.all(P[m] > 0.0)


def test_key_shift_invariance(oracle_mod):
    """k_j + c shifts every score in row i by scale*<q_i, c>: o unchanged."""
    N, d = 9, 6
    q = _randn((1, 1, N, 2, d), 11)
    k = _randn((1, 1, N, 1, d), 12)
    v = _randn((1, 1, N, 1, d), 13)
    c = _randn((d,), 14)
    scale = 1.0 / math.sqrt(d)
    o1, lse1 = oracle_mod.attn_fwd(q, k, v)
    o2, lse2 = oracle_mod.attn_fwd(q, k + c, v)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)
    shift = (q[0, 0] @ c).numpy().T * scale  # [Hq][N]
    np.testing.assert_allclose(lse2[0, 0] - lse1[0, 0], shift, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("P,N,Hq,Hkv,cu", [(2, 8, 4, 2, None), (4, 16, 8, 4, None),
                                           (2, 12, 4, 2, [0, 5, 12]), (4, 8, 8, 8, None)])
def test_ulysses_sharded_equals_unsharded(oracle_mod, P, N, Hq, Hkv, cu):
    """swap -> per-shard attention -> swap back == attention over all heads."""
    d, B = 4, 1
    q = _randn((P, B, N // P, Hq, d), 15)
    k = _randn((P, B, N // P, Hkv, d), 16)
    v = _randn((P, B, N // P, Hkv, d), 17)
    qh = oracle_mod.seq_to_head(q, P)
    kh = oracle_mod.seq_to_head(k, P)
    vh = oracle_mod.seq_to_head(v, P)
    oh, lse_h = oracle_mod.attn_fwd(qh, kh, vh, cu_seqlens=cu)
    o_seq = oracle_mod.head_to_seq(torch.from_numpy(oh), P)
    # unsharded: with B = 1 the P seq shards concatenated are [N][H][d]
    full = lambda x: x.reshape(1, B, N, x.shape[3], d)
    o_full, lse_full = oracle_mod.attn_fwd(full(q), full(k), full(v), cu_seqlens=cu)
    assert np.array_equal(o_seq.reshape(1, B, N, Hq, d).numpy(), o_full)
    # head shard r holds global heads [r*Hq/P, (r+1)*Hq/P)
    Hp = Hq // P
    for r in range(P):
        assert np.array_equal(lse_h[r, 0], lse_full[0, 0, r * Hp:(r + 1) * Hp])


def test_gqa_equals_repeated_kv(oracle_mod):
    N, d, Hq, Hkv = 10, 4, 6, 2
    q = _randn((1, 1, N, Hq, d), 18)
    k = _randn((1, 1, N, Hkv, d), 19)
    v = _randn((1, 1, N, Hkv, d), 20)
    o1, l1 = oracle_mod.attn_fwd(q, k, v)
    o2, l2 = oracle_mod.attn_fwd(q, k.repeat_interleave(Hq // Hkv, dim=3),
                                 v.repeat_interleave(Hq // Hkv, dim=3))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("causal", [True, False])
def test_packed_docs_equal_separate_docs(oracle_mod, causal):
    cu = [0, 4, 5, 11, 16]
    N, d = 16, 4
    q = _randn((1, 1, N, 2, d), 21)
    k = _randn((1, 1, N, 1, d), 22)
    v = _randn((1, 1, N, 1, d), 23)
    o, lse = oracle_mod.attn_fwd(q, k, v, causal=causal, cu_seqlens=cu)
    for a, b in zip(cu[:-1], cu[1:]):
        od, ld = oracle_mod.attn_fwd(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], causal=causal)
        assert np.array_equal(o[:, :, a:b], od)
        assert np.array_equal(lse[:, :, :, a:b], ld)


def test_rows_equal_full(oracle_mod):
    S, B, N, Hq, Hkv, d = 2, 1, 14, 4, 2, 4
    cu = [0, 6, 14]
    q = _randn((S, B, N, Hq, d), 24)
    k = _randn((S, B, N, Hkv, d), 25)
    v = _randn((S, B, N, Hkv, d), 26)
    o, lse = oracle_mod.attn_fwd(q, k, v, cu_seqlens=cu)
    rows = [(1, 0, 3, 13), (0, 0, 0, 0), (0, 0, 2, 6), (1, 0, 1, 5)]
    o_r, l_r = oracle_mod.attn_fwd_rows(q, k, v, rows, cu_seqlens=cu)
    for n, (s, b, h, i) in enumerate(rows):
        assert np.array_equal(o_r[n], o[s, b, i, h])
        assert l_r[n] == lse[s, b, h, i]
