"""GPU parity of the sequence-parallel loss: shifted labels across shard
boundaries, per-rank mean CE, good-token-weighted aggregation and the
gradient with respect to the logits, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity_utils import REL_TOL, Guards, log_errors, rel_fro

pytestmark = pytest.mark.gpu


def _case(P, B, N, V, dtype, seed, ignore_frac=0.25):
    g = torch.Generator().manual_seed(seed)
    Np = N // P
    logits = (torch.randn(P, B, Np, V, generator=g) * 2.0).to(dtype)
    labels = torch.randint(0, V, (P, B, Np), generator=g, dtype=torch.int64)
    labels[torch.rand(P, B, Np, generator=g) < ignore_frac] = -100
    return logits, labels


def _to_full(x, P):
    """[P][B][N/P](...) -> [B][N](...) : the unsharded sequence."""
    x = x.transpose(0, 1)
    return x.reshape(x.shape[0], -1, *x.shape[3:])


def _oracle(logits, labels, P):
    lf = _to_full(logits, P).double().numpy()
    yf = _to_full(labels, P).numpy()
    sh = oracle.shift_labels_batched(yf)
    losses, goods = oracle.per_rank_losses_batched(lf, sh, P)
    total = oracle.aggregate_sharded_loss(losses, goods)
    grad = oracle.aggregated_loss_grad(lf, sh, P)
    return np.array(losses), np.array(goods), total, grad


@pytest.mark.parametrize("P,B,N,V,dtype", [
    (4, 2, 64, 1000, torch.bfloat16),      # 16-byte vector path
    (4, 2, 64, 1000, torch.float32),
    (2, 1, 96, 1001, torch.bfloat16),      # V not a multiple of 8: scalar path
    (8, 3, 64, 257, torch.float32),
    (4, 1, 2048, 151936, torch.bfloat16),  # Qwen3 vocabulary: with the gradient, rows held by clusters of 4
    (4, 1, 128, 50000, torch.bfloat16),    # clusters of 2
    (2, 1, 256, 151936, torch.float32),    # clusters of 8
])
def test_sharded_ce_vs_oracle(uly, P, B, N, V, dtype):
    logits, labels = _case(P, B, N, V, dtype, seed=N + V)
    g = Guards()
    dl = g.empty(logits.shape, dtype, float("nan"))
    outs = (g.empty((P,), torch.float32), g.empty((P,), torch.int64), g.empty((1,), torch.float32))
    ws = g.workspace(uly.load().ulysses_sharded_ce_workspace_size(B, N, P))
    sl, sg, tot = uly.ulysses_sharded_ce_loss(logits.cuda(), labels.cuda(), P, dlogits=dl, workspace=ws,
                                              outputs=outs)
    torch.cuda.synchronize()
    assert uly.ulysses_get_device_status()[0] == 0
    g.check()
    losses, goods, total, grad = _oracle(logits, labels, P)
    assert sg.cpu().numpy().tolist() == goods.tolist()
    tag = "bf16" if dtype == torch.bfloat16 else "fp32"
    loss_err = float(np.max(np.abs(sl.cpu().double().numpy() - losses) / np.maximum(np.abs(losses), 1e-12)))
    tot_err = abs(float(tot.cpu()) - total) / abs(total)
    grad_full = _to_full(dl.cpu(), P)
    gerr = rel_fro(grad_full, grad)
    log_errors(f"sharded ce P{P} B{B} N{N} V{V} {tag}", shard_loss_rel=loss_err, total_rel=tot_err, dlogits=gerr)
    assert loss_err <= 1e-5 and tot_err <= 1e-5, (loss_err, tot_err)
    assert gerr <= REL_TOL[tag], gerr


def test_last_token_of_a_shard_targets_the_next_shard(uly):
    """Shifting after sharding would drop P-1 targets; the kernel keeps them."""
    P, B, N, V = 4, 1, 32, 64
    logits, labels = _case(P, B, N, V, torch.float32, seed=3, ignore_frac=0.0)
    sl, sg, tot = uly.ulysses_sharded_ce_loss(logits.cuda(), labels.cuda(), P)
    torch.cuda.synchronize()
    assert sg.cpu().tolist() == [N // P] * (P - 1) + [N // P - 1]


def test_all_ignored_and_invalid_labels(uly):
    P, B, N, V = 2, 1, 16, 32
    logits, labels = _case(P, B, N, V, torch.float32, seed=4)
    labels[:] = -100
    dl = torch.full(logits.shape, float("nan"), device="cuda")
    sl, sg, tot = uly.ulysses_sharded_ce_loss(logits.cuda(), labels.cuda(), P, dlogits=dl)
    torch.cuda.synchronize()
    assert sg.cpu().tolist() == [0, 0] and float(tot.cpu()) == 0.0 and sl.cpu().tolist() == [0.0, 0.0]
    assert float(dl.abs().max()) == 0.0
    assert uly.ulysses_get_device_status()[0] == 0
    labels[0, 0, 3] = V + 5  # out of range: ignored and reported
    uly.ulysses_sharded_ce_loss(logits.cuda(), labels.cuda(), P)
    assert uly.ulysses_get_device_status()[0] == 1   # ULY_ERR_INVALID_ARG


def _random_loss_cases(n, seed=31):
    """Seeded random loss shapes: P in 1..8, batches, vocabularies from a few
    entries to beyond Qwen3's (multiples of 8 or not: vector and scalar paths,
    every cluster size), both dtypes."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        P = int(rng.choice([1, 2, 4, 8]))
        N = P * int(rng.integers(1, 64 // P + 2))
        V = int(rng.choice([int(rng.integers(2, 600)), int(rng.integers(1000, 200000))]))
        if rng.integers(0, 2) and V >= 8:
            V -= V % 8  # a multiple of 8: the 16-byte vector path (clusters with the gradient)
        dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
        out.append((P, int(rng.integers(1, 3)), N, V, dtype))
    return out


@pytest.mark.parametrize("P,B,N,V,dtype", _random_loss_cases(6))
def test_sharded_ce_random_shapes(uly, P, B, N, V, dtype):
    test_sharded_ce_vs_oracle(uly, P, B, N, V, dtype)
