"""Good-token-weighted loss aggregation across sequence-parallel ranks (fp64).

TEST INFRASTRUCTURE ONLY (part of the oracle).

Follows the Accelerate PR "Deepspeed Ulysses/ALST integration" (user API,
step 2): labels are shifted over the full sequence before sharding, every
rank computes the mean cross entropy over its own tokens whose label is not
-100, and the ranks' losses are combined weighted by their good-token counts,
divided by max(total good tokens, 1).

Reading where the page is silent: a rank with no good tokens reports loss 0
(its weight is 0 anyway; an empty mean would otherwise be NaN and 0 * NaN is
NaN).
"""
from __future__ import annotations

import numpy as np

IGNORE = -100


def shift_labels(labels: np.ndarray) -> np.ndarray:
    """Next-token labels over the whole sequence: out[i] = labels[i+1], last = -100."""
    labels = np.asarray(labels, dtype=np.int64)
    out = np.full_like(labels, IGNORE)
    out[:-1] = labels[1:]
    return out


def _token_ce(logits: np.ndarray, label: int) -> float:
    row = np.asarray(logits, dtype=np.float64)
    m = row.max()
    lse = m + np.log(np.exp(row - m).sum())
    return float(lse - row[label])


def per_rank_losses(logits: np.ndarray, shifted: np.ndarray, P: int):
    """Split tokens into P contiguous shards; per shard mean CE and good count."""
    N = len(shifted)
    assert N % P == 0, "sequence must be padded to a multiple of the SP size"
    Np = N // P
    losses, goods = [], []
    for r in range(P):
        total, good = 0.0, 0
        for i in range(r * Np, (r + 1) * Np):
            if shifted[i] != IGNORE:
                total += _token_ce(logits[i], int(shifted[i]))
                good += 1
        losses.append(total / good if good > 0 else 0.0)
        goods.append(good)
    return losses, goods


def aggregate_sharded_loss(losses, goods) -> float:
    """sum_r loss_r * good_r / max(sum_r good_r, 1)."""
    total = 0.0
    for loss_r, good_r in zip(losses, goods):
        total += loss_r * good_r
    return total / max(sum(goods), 1)


def full_sequence_loss(logits: np.ndarray, shifted: np.ndarray) -> float:
    """Mean CE over all good tokens of the unsharded sequence (0 if none)."""
    total, good = 0.0, 0
    for i in range(len(shifted)):
        if shifted[i] != IGNORE:
            total += _token_ce(logits[i], int(shifted[i]))
            good += 1
    return total / max(good, 1)
