"""Pins for the oracle's attention backward (CPU only).

* central finite differences of L = sum(O * dO) on tiny fp64 inputs;
* torch fp64 autograd through an explicit masked softmax attention;
* exact invariants: sum_j dV_j = sum over the GQA group of sum_i dO_i
  (softmax rows sum to 1) and sum_j dK_j = 0 (sum_j dS_ij = 0);
* sampled dq / dk / dv rows equal the full backward;
* Ulysses-sharded gradients equal unsharded gradients.
"""
import math

import numpy as np
import pytest
import torch


def _randn(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


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


def _loss(oracle_mod, q, k, v, dout, causal, cu):
    o, _ = oracle_mod.attn_fwd(q, k, v, causal=causal, cu_seqlens=cu)
    return float((o * dout.numpy()).sum())


@pytest.mark.parametrize("causal,cu", [(True, None), (False, None), (True, [0, 3, 4, 9])])
def test_finite_differences(oracle_mod, causal, cu):
    N, Hq, Hkv, d = 9, 2, 1, 4
    q = _randn((1, 1, N, Hq, d), 1)
    k = _randn((1, 1, N, Hkv, d), 2)
    v = _randn((1, 1, N, Hkv, d), 3)
    do = _randn((1, 1, N, Hq, d), 4)
    dq, dk, dv, _, _ = oracle_mod.attn_bwd(q, k, v, do, causal=causal, cu_seqlens=cu)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(g)
        flat = x.view(-1)
        for idx in range(flat.numel()):
            old = float(flat[idx])
            flat[idx] = old + h
            lp = _loss(oracle_mod, q, k, v, do, causal, cu)
            flat[idx] = old - h
            lm = _loss(oracle_mod, q, k, v, do, causal, cu)
            flat[idx] = old
            num.reshape(-1)[idx] = (lp - lm) / (2 * h)
        rel = np.linalg.norm(num - g) / np.linalg.norm(g)
        assert rel <= 1e-6, (name, rel)


@pytest.mark.parametrize("S,B,N,Hq,Hkv,d,causal,cu", [
    (1, 1, 12, 4, 2, 8, True, None),
    (2, 2, 10, 2, 1, 4, False, None),
    (1, 1, 17, 4, 1, 4, True, [0, 7, 8, 17]),
    (1, 1, 15, 2, 1, 4, False, [0, 0, 6, 6, 15, 15]),  # zero-length documents
])
def test_matches_torch_autograd(oracle_mod, S, B, N, Hq, Hkv, d, causal, cu):
    q = _randn((S, B, N, Hq, d), 5).requires_grad_()
    k = _randn((S, B, N, Hkv, d), 6).requires_grad_()
    v = _randn((S, B, N, Hkv, d), 7).requires_grad_()
    do = _randn((S, B, N, Hq, d), 8)
    scale = 1.0 / math.sqrt(d)
    G = Hq // Hkv
    mask = _mask(N, causal, cu)
    kk = k.repeat_interleave(G, dim=3)
    vv = v.repeat_interleave(G, dim=3)
    s = torch.einsum("sbihd,sbjhd->sbhij", q, kk) * scale
    p = torch.softmax(s.masked_fill(~mask, -math.inf), dim=-1)
    o = torch.einsum("sbhij,sbjhd->sbihd", p, vv)
    (o * do).sum().backward()
    dq, dk, dv, o_or, lse = oracle_mod.attn_bwd(q.detach(), k.detach(), v.detach(), do,
                                                causal=causal, cu_seqlens=cu)
    np.testing.assert_allclose(o_or, o.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("causal,cu", [(True, None), (True, [0, 10, 13, 24])])
def test_sum_invariants(oracle_mod, causal, cu):
    S, B, N, Hq, Hkv, d = 2, 1, 24, 4, 2, 8
    q = _randn((S, B, N, Hq, d), 9)
    k = _randn((S, B, N, Hkv, d), 10)
    v = _randn((S, B, N, Hkv, d), 11)
    do = _randn((S, B, N, Hq, d), 12)
    dq, dk, dv, _, _ = oracle_mod.attn_bwd(q, k, v, do, causal=causal, cu_seqlens=cu)
    G = Hq // Hkv
    for s in range(S):
        for kvh in range(Hkv):
            sum_dv = dv[s, 0, :, kvh].sum(0)
            sum_do = do[s, 0, :, kvh * G:(kvh + 1) * G].sum((0, 1)).numpy()
            np.testing.assert_allclose(sum_dv, sum_do, rtol=1e-12, atol=1e-12)
            assert np.abs(dk[s, 0, :, kvh].sum(0)).max() <= 1e-12


def test_rows_equal_full(oracle_mod):
    S, B, N, Hq, Hkv, d = 2, 2, 15, 4, 2, 4
    cu = [0, 8, 15]
    q = _randn((S, B, N, Hq, d), 13)
    k = _randn((S, B, N, Hkv, d), 14)
    v = _randn((S, B, N, Hkv, d), 15)
    do = _randn((S, B, N, Hq, d), 16)
    dq, dk, dv, _, _ = oracle_mod.attn_bwd(q, k, v, do, cu_seqlens=cu)
    rows = [(1, 1, 3, 14), (0, 0, 0, 0), (0, 1, 2, 7), (1, 0, 1, 9)]
    dq_r = oracle_mod.attn_bwd_q_rows(q, k, v, do, rows, cu_seqlens=cu)
    for n, (s, b, h, i) in enumerate(rows):
        np.testing.assert_allclose(dq_r[n], dq[s, b, i, h], rtol=1e-13, atol=1e-14)
    # keys sharing their attending rows (same shard, batch and KV head) and
    # one repeated key: each row's forward is computed once and every key sums
    # over its rows as the full backward does, so the rows are bit-identical
    keys = [(1, 1, 1, 14), (0, 0, 0, 0), (0, 1, 1, 8), (1, 0, 0, 3), (1, 0, 0, 5), (1, 0, 0, 3)]
    dk_r, dv_r = oracle_mod.attn_bwd_kv_rows(q, k, v, do, keys, cu_seqlens=cu)
    for n, (s, b, kvh, j) in enumerate(keys):
        assert np.array_equal(dk_r[n], dk[s, b, j, kvh]), (n, dk_r[n], dk[s, b, j, kvh])
        assert np.array_equal(dv_r[n], dv[s, b, j, kvh]), (n, dv_r[n], dv[s, b, j, kvh])


@pytest.mark.parametrize("causal", [True, False])
def test_kv_rows_of_one_group_equal_full(oracle_mod, causal):
    """Every key of one (shard, batch, KV head), so all attending rows are
    shared between keys: still the full backward's rows bit for bit."""
    S, B, N, Hq, Hkv, d = 1, 1, 21, 6, 2, 4
    q = _randn((S, B, N, Hq, d), 21)
    k = _randn((S, B, N, Hkv, d), 22)
    v = _randn((S, B, N, Hkv, d), 23)
    do = _randn((S, B, N, Hq, d), 24)
    dq, dk, dv, _, _ = oracle_mod.attn_bwd(q, k, v, do, causal=causal)
    keys = [(0, 0, 1, j) for j in range(N)]
    dk_r, dv_r = oracle_mod.attn_bwd_kv_rows(q, k, v, do, keys, causal=causal)
    assert np.array_equal(dk_r, dk[0, 0, :, 1])
    assert np.array_equal(dv_r, dv[0, 0, :, 1])


def test_ulysses_sharded_grads_equal_unsharded(oracle_mod):
    """dO goes seq->head, gradients come back head->seq (the inverse swaps)."""
    P, B, N, Hq, Hkv, d = 2, 1, 10, 4, 2, 4
    q = _randn((P, B, N // P, Hq, d), 17)
    k = _randn((P, B, N // P, Hkv, d), 18)
    v = _randn((P, B, N // P, Hkv, d), 19)
    do = _randn((P, B, N // P, Hq, d), 20)
    sh = lambda x: oracle_mod.seq_to_head(x, P)
    dq_h, dk_h, dv_h, _, _ = oracle_mod.attn_bwd(sh(q), sh(k), sh(v), sh(do))
    back = lambda x: oracle_mod.head_to_seq(torch.from_numpy(x), P).reshape(1, B, N, -1, d).numpy()
    full = lambda x: x.reshape(1, B, N, x.shape[3], d)
    dq, dk, dv, _, _ = oracle_mod.attn_bwd(full(q), full(k), full(v), full(do))
    np.testing.assert_allclose(back(dq_h), dq, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(back(dk_h), dk, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(back(dv_h), dv, rtol=1e-13, atol=1e-14)
