"""Ring attention (P chunks meeting in P ring steps, merged through their
log-sum-exp) against the fp64 oracle's plain causal attention, and against
the Ulysses path that computes the same function with head sharding."""
import numpy as np
import pytest
import torch

import oracle
from parity_utils import LSE_TOL, REL_TOL, Guards, log_errors, max_abs, rel_fro
from ulysses_inputs import WORKLOADS, draw_seq_inputs

pytestmark = pytest.mark.gpu


def _ring(uly, seq, P, causal=True):
    q, k, v, do = (seq[n].cuda() for n in ("q", "k", "v", "dout"))
    Ps, B, Np, Hq, d = q.shape
    Hkv = k.shape[3]
    g = Guards()
    o = g.full_like(q, float("nan"))
    lse = g.empty((P, B, Hq, Np), torch.float32, float("nan"))
    dt = 0 if q.dtype == torch.bfloat16 else 1
    ws_f = g.workspace(uly.load().ulysses_ring_attn_workspace_size(B, Np * P, Hq, Hkv, d, P, 0, dt))
    uly.ulysses_ring_attn_fwd(q, k, v, o, lse, P, causal=causal, workspace=ws_f)
    dq, dk, dv = (g.full_like(x, float("nan")) for x in (q, k, v))
    ws_b = g.workspace(uly.load().ulysses_ring_attn_workspace_size(B, Np * P, Hq, Hkv, d, P, 1, dt))
    uly.ulysses_ring_attn_bwd(q, k, v, o, lse, do, dq, dk, dv, P, causal=causal, workspace=ws_b)
    torch.cuda.synchronize()
    assert uly.ulysses_get_device_status()[0] == 0
    g.check()
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


def _oracle_full(seq, causal):
    """Attention over all heads of the unsharded sequence (B = 1): [1][1][N][H][d]."""
    full = lambda x: x.reshape(1, 1, -1, x.shape[3], x.shape[4])
    dq, dk, dv, o, lse = oracle.attn_bwd(full(seq["q"]), full(seq["k"]), full(seq["v"]), full(seq["dout"]),
                                         causal=causal)
    return dq, dk, dv, o, lse


@pytest.mark.parametrize("name,N,P,causal", [
    ("tiny_fp32_n256", None, None, True),
    ("qwen3_4b_n8192", 512, 4, True),
    ("qwen3_4b_n8192", 400, 4, True),     # chunks of 100 tokens: ragged tiles
    ("qwen3_4b_n8192", 384, 3, False),    # non-causal: the wrapped pairs too
    ("qwen3_4b_n8192", 256, 1, True),     # one rank: plain attention
])
def test_ring_vs_oracle(uly, name, N, P, causal):
    w = WORKLOADS[name]
    P = P or w.P
    seq = draw_seq_inputs(w, seed=12, N=N, P=P)
    r = _ring(uly, seq, P, causal)
    dq, dk, dv, o, lse = _oracle_full(seq, causal)
    Nn = o.shape[2]
    Np = Nn // P
    seqv = lambda t: t.reshape(-1, t.shape[3], t.shape[4]).cpu()   # [N][H][d]
    tag = w.dtype
    errs = dict(o=rel_fro(seqv(r["o"]), o[0, 0]), dq=rel_fro(seqv(r["dq"]), dq[0, 0]),
                dk=rel_fro(seqv(r["dk"]), dk[0, 0]), dv=rel_fro(seqv(r["dv"]), dv[0, 0]))
    # lse [P][B][Hq][Np] -> [Hq][N]
    lse_g = r["lse"][:, 0].permute(1, 0, 2).reshape(lse.shape[2], Nn).cpu()
    errs["lse_max_abs"] = max_abs(lse_g, lse[0, 0])
    log_errors(f"ring {name} N{Nn} P{P} causal{int(causal)}", **errs)
    for key in ("o", "dq", "dk", "dv"):
        assert errs[key] <= REL_TOL[tag], errs
    assert errs["lse_max_abs"] <= LSE_TOL[tag], errs


def test_ring_equals_ulysses_path(uly):
    """Ring attention and the Ulysses path compute the same function."""
    w = WORKLOADS["qwen3_4b_n8192"]
    P, N = 4, 1024
    seq = draw_seq_inputs(w, seed=13, N=N)
    r = _ring(uly, seq, P)
    q, k, v, do = (seq[n].cuda() for n in ("q", "k", "v", "dout"))
    o = torch.empty_like(q)
    lse = torch.empty(P, 1, w.Hq // P, N, dtype=torch.float32, device="cuda")
    uly.ulysses_attn_fwd_seq(q, k, v, o, lse, P)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    uly.ulysses_attn_bwd_seq(q, k, v, o, lse, do, dq, dk, dv, P)
    torch.cuda.synchronize()
    for a, b, name in ((r["o"], o, "o"), (r["dq"], dq, "dq"), (r["dk"], dk, "dk"), (r["dv"], dv, "dv")):
        assert rel_fro(a, b) <= REL_TOL["bf16"], name


def test_ring_bench_workload_sampled(uly, oracle_mod):
    """The 65536-token workload through ring attention, sampled rows vs the oracle."""
    w = WORKLOADS["qwen3_4b_n65536"]
    seq = draw_seq_inputs(w, seed=14, device="cuda")
    r = _ring(uly, seq, w.P)
    oh = {n: oracle_mod.seq_to_head(seq[n].cpu(), w.P) for n in seq}
    rng = np.random.default_rng(8)
    rows = [(int(rng.integers(w.P)), 0, int(rng.integers(w.Hp)), int(rng.integers(w.N))) for _ in range(32)]
    o_ref, lse_ref = oracle_mod.attn_fwd_rows(oh["q"], oh["k"], oh["v"], rows)
    dq_ref = oracle_mod.attn_bwd_q_rows(oh["q"], oh["k"], oh["v"], oh["dout"], rows[:12])
    Np = w.N // w.P

    def seq_row(t, s, h, i):  # head shard s, local head h, token i -> [chunk][0][pos][global head]
        return t[i // Np, 0, i % Np, s * w.Hp + h].double().cpu().numpy()
    o_gpu = np.stack([seq_row(r["o"], s, h, i) for s, b, h, i in rows])
    dq_gpu = np.stack([seq_row(r["dq"], s, h, i) for s, b, h, i in rows[:12]])
    lse_gpu = np.array([float(r["lse"][i // Np, 0, s * w.Hp + h, i % Np]) for s, b, h, i in rows])
    errs = dict(o=rel_fro(o_gpu, o_ref), dq=rel_fro(dq_gpu, dq_ref), lse_max_abs=float(np.abs(lse_gpu - lse_ref).max()))
    log_errors("ring qwen3_4b_n65536 sampled", **errs)
    assert errs["o"] <= REL_TOL["bf16"] and errs["dq"] <= REL_TOL["bf16"], errs
    assert errs["lse_max_abs"] <= LSE_TOL["bf16"], errs


def _random_ring_cases(n, seed=55):
    """Seeded random ring shapes with the Qwen3-4B head counts: P a divisor
    of the 8 KV heads (1, 2, 4, 8), N a multiple of P with ragged chunks,
    causal or not."""
    import numpy as np
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        P = int(rng.choice([1, 2, 4, 8]))
        out.append(("qwen3_4b_n8192", P * int(rng.integers(20, 160)), P, bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("name,N,P,causal", _random_ring_cases(4))
def test_ring_random_shapes_vs_oracle(uly, name, N, P, causal):
    test_ring_vs_oracle(uly, name, N, P, causal)
