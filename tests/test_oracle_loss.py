"""Pins for the oracle's good-token-weighted loss aggregation (CPU only).

The aggregation of per-rank mean losses weighted by good-token counts must
equal the mean over the good tokens of the whole (unsharded) sequence, which
torch's ``cross_entropy(ignore_index=-100)`` computes independently.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from ulysses_inputs import draw_labels_logits


def _torch_mean_ce(logits, shifted):
    lt = torch.from_numpy(logits)
    yt = torch.from_numpy(shifted)
    if (yt != -100).sum() == 0:
        return 0.0
    return float(F.cross_entropy(lt, yt, ignore_index=-100, reduction="mean"))


def test_shift_labels(oracle_mod):
    lab = np.array([5, 6, -100, 7, 8, 9], dtype=np.int64)
    assert oracle_mod.shift_labels(lab).tolist() == [6, -100, 7, 8, 9, -100]


@pytest.mark.parametrize("N,V,P,frac,seed", [(16, 7, 4, 0.3, 0), (24, 5, 2, 0.6, 1),
                                             (32, 11, 8, 0.0, 2), (12, 3, 4, 0.9, 3)])
def test_aggregate_equals_full_mean(oracle_mod, N, V, P, frac, seed):
    logits, labels = draw_labels_logits(N, V, seed, ignore_frac=frac)
    shifted = oracle_mod.shift_labels(labels)
    losses, goods = oracle_mod.per_rank_losses(logits, shifted, P)
    agg = oracle_mod.aggregate_sharded_loss(losses, goods)
    assert agg == pytest.approx(oracle_mod.full_sequence_loss(logits, shifted), rel=1e-13, abs=1e-15)
    assert agg == pytest.approx(_torch_mean_ce(logits, shifted), rel=1e-12, abs=1e-15)


def test_empty_rank_and_all_ignored(oracle_mod):
    N, V, P = 16, 6, 4
    logits, labels = draw_labels_logits(N, V, 7, ignore_frac=0.0)
    labels[: N // P + 1] = -100  # rank 0 has no good token after the shift
    shifted = oracle_mod.shift_labels(labels)
    losses, goods = oracle_mod.per_rank_losses(logits, shifted, P)
    assert goods[0] == 0 and losses[0] == 0.0
    agg = oracle_mod.aggregate_sharded_loss(losses, goods)
    assert agg == pytest.approx(_torch_mean_ce(logits, shifted), rel=1e-12)
    # all ignored: 0 / max(0, 1) = 0
    none = np.full(N, -100, dtype=np.int64)
    l2, g2 = oracle_mod.per_rank_losses(logits, none, P)
    assert oracle_mod.aggregate_sharded_loss(l2, g2) == 0.0


def test_shift_before_sharding_crosses_boundaries(oracle_mod):
    """The label of the last token of a shard is the first token of the next."""
    N, V, P = 8, 4, 2
    logits, labels = draw_labels_logits(N, V, 11, ignore_frac=0.0)
    shifted = oracle_mod.shift_labels(labels)
    assert shifted[N // P - 1] == labels[N // P]
    # sharding first and shifting inside each shard would lose that target
    losses, goods = oracle_mod.per_rank_losses(logits, shifted, P)
    assert sum(goods) == N - 1


def test_batched_reduces_to_single_row(oracle_mod):
    N, V, P = 16, 5, 4
    logits, labels = draw_labels_logits(N, V, 21, ignore_frac=0.2)
    sh = oracle_mod.shift_labels(labels)
    l1, g1 = oracle_mod.per_rank_losses(logits, sh, P)
    l2, g2 = oracle_mod.per_rank_losses_batched(logits[None], oracle_mod.shift_labels_batched(labels[None]), P)
    assert g1 == g2 and np.allclose(l1, l2, rtol=0, atol=0)


def test_batched_aggregate_equals_torch_mean(oracle_mod):
    B, N, V, P = 3, 12, 7, 4
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((B, N, V))
    labels = rng.integers(0, V, size=(B, N))
    labels[rng.random((B, N)) < 0.3] = -100
    sh = oracle_mod.shift_labels_batched(labels)
    losses, goods = oracle_mod.per_rank_losses_batched(logits, sh, P)
    agg = oracle_mod.aggregate_sharded_loss(losses, goods)
    ref = F.cross_entropy(torch.from_numpy(logits).reshape(-1, V), torch.from_numpy(sh).reshape(-1),
                          ignore_index=-100, reduction="mean")
    assert agg == pytest.approx(float(ref), rel=1e-12)


def test_aggregated_grad_matches_autograd_and_finite_differences(oracle_mod):
    B, N, V, P = 2, 8, 5, 2
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((B, N, V))
    labels = rng.integers(0, V, size=(B, N))
    labels[0, 2] = -100
    sh = oracle_mod.shift_labels_batched(labels)
    g = oracle_mod.aggregated_loss_grad(logits, sh, P)
    lt = torch.from_numpy(logits.copy()).requires_grad_()
    F.cross_entropy(lt.reshape(-1, V), torch.from_numpy(sh).reshape(-1), ignore_index=-100).backward()
    np.testing.assert_allclose(g, lt.grad.numpy(), rtol=1e-12, atol=1e-14)

    def total(x):
        l, c = oracle_mod.per_rank_losses_batched(x, sh, P)
        return oracle_mod.aggregate_sharded_loss(l, c)
    h = 1e-6
    for idx in [(0, 0, 1), (1, 5, 4), (0, 7, 0), (0, 2, 3)]:
        x = logits.copy(); x[idx] += h
        y = logits.copy(); y[idx] -= h
        assert (total(x) - total(y)) / (2 * h) == pytest.approx(g[idx], abs=1e-8)
