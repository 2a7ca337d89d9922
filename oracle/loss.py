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


# ------------------------------------------------------------------ batched
# The Trainer shards every row of the local batch the same way: rank r holds
# tokens [r*N/P, (r+1)*N/P) of each of the B rows, and its loss is the mean
# over all of its good tokens (all rows).

def shift_labels_batched(labels: np.ndarray) -> np.ndarray:
    """labels [B][N] -> next-token labels per row, last of each row -100."""
    labels = np.asarray(labels, dtype=np.int64)
    return np.stack([shift_labels(row) for row in labels])


def per_rank_losses_batched(logits: np.ndarray, shifted: np.ndarray, P: int):
    """logits [B][N][V], shifted [B][N] -> per-rank mean CE and good counts."""
    B, N = shifted.shape
    assert N % P == 0
    Np = N // P
    losses, goods = [], []
    for r in range(P):
        total, good = 0.0, 0
        for b in range(B):
            for i in range(r * Np, (r + 1) * Np):
                if shifted[b, i] != IGNORE:
                    total += _token_ce(logits[b, i], int(shifted[b, i]))
                    good += 1
        losses.append(total / good if good > 0 else 0.0)
        goods.append(good)
    return losses, goods


def aggregated_loss_grad(logits: np.ndarray, shifted: np.ndarray, P: int) -> np.ndarray:
    """Gradient of the aggregated loss with respect to logits [B][N][V].

    total = sum_r loss_r * good_r / max(T, 1) with loss_r = (sum of CE over
    rank r's good tokens) / good_r, so total = (sum of CE over all good
    tokens) / max(T, 1) and d total / d logit[b, i, :] = (softmax(logit[b,i]) -
    onehot(label)) / max(T, 1) for good tokens, 0 for ignored ones.
    """
    logits = np.asarray(logits, dtype=np.float64)
    B, N, V = logits.shape
    T = int((shifted != IGNORE).sum())
    g = np.zeros_like(logits)
    for b in range(B):
        for i in range(N):
            y = int(shifted[b, i])
            if y == IGNORE:
                continue
            row = logits[b, i]
            e = np.exp(row - row.max())
            g[b, i] = e / e.sum()
            g[b, i, y] -= 1.0
            g[b, i] /= max(T, 1)
    return g
