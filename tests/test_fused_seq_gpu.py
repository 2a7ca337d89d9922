"""The fused seq-layout attention (no swaps) against the oracle and against
the three-step path swap -> attention -> swap it replaces."""
import numpy as np
import pytest
import torch

import oracle
from parity_utils import LSE_TOL, REL_TOL, Guards, bytes_equal, log_errors, max_abs, rel_fro
from ulysses_inputs import WORKLOADS, cu_seqlens_from_lengths, draw_seq_inputs

pytestmark = pytest.mark.gpu


def _run_fused(uly, seq, P, cu=None):
    q, k, v, do = (seq[n].cuda() for n in ("q", "k", "v", "dout"))
    Ps, B, Np, Hq, d = q.shape
    N = Np * P
    g = Guards()
    o = g.full_like(q, float("nan"))
    lse = g.empty((P, B, Hq // P, N), torch.float32, float("nan"))
    uly.ulysses_attn_fwd_seq(q, k, v, o, lse, P, cu_seqlens=cu)
    dq, dk, dv = (g.full_like(x, float("nan")) for x in (q, k, v))
    uly.ulysses_attn_bwd_seq(q, k, v, o, lse, do, dq, dk, dv, P, cu_seqlens=cu)
    torch.cuda.synchronize()
    assert uly.ulysses_get_device_status()[0] == 0
    g.check()
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


@pytest.mark.parametrize("name,N,P,cu", [
    ("tiny_fp32_n256", None, None, None),
    ("qwen3_4b_n8192", 1024, 4, None),
    ("qwen3_4b_n8192", 1024, 2, [0, 100, 612, 613, 1024]),   # docs crossing shard boundaries
    ("qwen3_4b_n8192", 2048, 8, None),
])
def test_fused_vs_oracle(uly, oracle_mod, name, N, P, cu):
    w = WORKLOADS[name]
    P = P or w.P
    seq = draw_seq_inputs(w, seed=9, N=N, P=P)
    tag = w.dtype
    r = _run_fused(uly, seq, P, cu)
    oh = {n: oracle_mod.seq_to_head(seq[n], P) for n in seq}
    dq, dk, dv, o, lse = oracle_mod.attn_bwd(oh["q"], oh["k"], oh["v"], oh["dout"], cu_seqlens=cu)
    back = lambda x: oracle_mod.head_to_seq(torch.from_numpy(x), P)
    errs = dict(o=rel_fro(r["o"], back(o)), dq=rel_fro(r["dq"], back(dq)), dk=rel_fro(r["dk"], back(dk)),
                dv=rel_fro(r["dv"], back(dv)), lse_max_abs=max_abs(r["lse"], lse))
    log_errors(f"fused seq {name} N{N} P{P} docs{0 if cu is None else len(cu) - 1}", **errs)
    for key in ("o", "dq", "dk", "dv"):
        assert errs[key] <= REL_TOL[tag], errs
    assert errs["lse_max_abs"] <= LSE_TOL[tag], errs


def test_fused_equals_three_step_path(uly):
    """Same arithmetic in the same order: O, lse, dK, dV bit for bit; dQ up to
    the order of its fp32 reductions."""
    w = WORKLOADS["qwen3_4b_n8192"]
    P, N = 4, 2048
    seq = draw_seq_inputs(w, seed=4, N=N)
    r = _run_fused(uly, seq, P)
    q, k, v, do = (seq[n].cuda() for n in ("q", "k", "v", "dout"))
    head = {}
    for n, x in (("q", q), ("k", k), ("v", v), ("dout", do)):
        head[n] = torch.empty(P, 1, N, x.shape[3] // P, 128, dtype=x.dtype, device="cuda")
        uly.ulysses_seq_to_head(x, head[n], P)
    o = torch.empty_like(head["q"])
    lse = torch.empty(P, 1, w.Hq // P, N, dtype=torch.float32, device="cuda")
    uly.ulysses_attn_fwd(head["q"], head["k"], head["v"], o, lse)
    dq, dk, dv = (torch.empty_like(head[n]) for n in ("q", "k", "v"))
    uly.ulysses_attn_bwd(head["q"], head["k"], head["v"], o, lse, head["dout"], dq, dk, dv)
    outs = {}
    for n, x, H in (("o", o, w.Hq), ("dq", dq, w.Hq), ("dk", dk, w.Hkv), ("dv", dv, w.Hkv)):
        outs[n] = torch.empty(P, 1, N // P, H, 128, dtype=x.dtype, device="cuda")
        uly.ulysses_head_to_seq(x, outs[n], P)
    torch.cuda.synchronize()
    assert bytes_equal(r["o"], outs["o"])
    assert bytes_equal(r["lse"], lse)
    assert bytes_equal(r["dk"], outs["dk"])
    assert bytes_equal(r["dv"], outs["dv"])
    assert rel_fro(r["dq"], outs["dq"]) <= 1e-3


def test_fused_bench_workload_sampled(uly, oracle_mod):
    """The 65536-token workload through the fused calls, sampled rows vs the oracle."""
    w = WORKLOADS["qwen3_4b_n65536"]
    seq = draw_seq_inputs(w, seed=6, device="cuda")
    r = _run_fused(uly, seq, w.P)
    oh = {n: oracle_mod.seq_to_head(seq[n].cpu(), w.P) for n in seq}
    rng = np.random.default_rng(5)
    rows = [(int(rng.integers(w.P)), 0, int(rng.integers(w.Hp)), int(rng.integers(w.N))) for _ in range(32)]
    o_ref, lse_ref = oracle_mod.attn_fwd_rows(oh["q"], oh["k"], oh["v"], rows)
    dq_ref = oracle_mod.attn_bwd_q_rows(oh["q"], oh["k"], oh["v"], oh["dout"], rows[:12])
    Np = w.N // w.P

    def seq_row(t, s, h, i):  # head shard s, local head h, token i -> seq-layout row
        return t[i // Np, 0, i % Np, s * (t.shape[3] // w.P) + h]
    o_gpu = np.stack([seq_row(r["o"], s, h, i).double().cpu().numpy() for s, b, h, i in rows])
    dq_gpu = np.stack([seq_row(r["dq"], s, h, i).double().cpu().numpy() for s, b, h, i in rows[:12]])
    lse_gpu = np.array([float(r["lse"][s, b, h, i]) for s, b, h, i in rows])
    errs = dict(o=rel_fro(o_gpu, o_ref), dq=rel_fro(dq_gpu, dq_ref), lse_max_abs=float(np.abs(lse_gpu - lse_ref).max()))
    log_errors("fused seq qwen3_4b_n65536 sampled", **errs)
    assert errs["o"] <= REL_TOL["bf16"] and errs["dq"] <= REL_TOL["bf16"], errs
    assert errs["lse_max_abs"] <= LSE_TOL["bf16"], errs


def _random_fused_cases(n, seed=77):
    """Seeded random fused-layout shapes with the Qwen3-4B head counts: P in
    {1, 2, 4, 8}, N/P a multiple of 128 (the bf16 path's requirement), and
    documents whose boundaries fall anywhere (across shard boundaries too)."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        P = int(rng.choice([1, 2, 4, 8]))
        N = P * 128 * int(rng.integers(1, max(2, 1536 // (P * 128) + 1)))
        cu = None
        if i % 2 == 0:
            cuts = sorted(set(int(c) for c in rng.integers(1, N, size=int(rng.integers(1, 5)))))
            cu = [0] + cuts + [N]
        out.append((N, P, cu))
    return out


@pytest.mark.parametrize("N,P,cu", _random_fused_cases(4))
def test_fused_random_shapes_vs_oracle(uly, oracle_mod, N, P, cu):
    test_fused_vs_oracle(uly, oracle_mod, "qwen3_4b_n8192", N, P, cu)
