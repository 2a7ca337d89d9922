"""GPU parity of attention forward/backward against the fp64 oracle, element
by element, at sizes that span several 128-row tiles with a ragged tail, plus
the degenerate cases (one token, one-token documents, odd GQA groups,
non-causal, packed documents) and the full fp32 workload through every step.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity_utils import LSE_TOL, REL_TOL, bytes_equal, log_errors, max_abs, rel_fro, run_path
from ulysses_inputs import WORKLOADS, draw_seq_inputs

pytestmark = pytest.mark.gpu


def _rand(shape, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


def _attn_case(uly, S, B, N, Hq, Hkv, d, dtype, causal, cu, seed=0):
    tag = "bf16" if dtype == torch.bfloat16 else "fp32"
    q = _rand((S, B, N, Hq, d), seed + 1, dtype)
    k = _rand((S, B, N, Hkv, d), seed + 2, dtype)
    v = _rand((S, B, N, Hkv, d), seed + 3, dtype)
    do = _rand((S, B, N, Hq, d), seed + 4, dtype)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((S, B, Hq, N), float("nan"), dtype=torch.float32, device="cuda")
    uly.ulysses_attn_fwd(qd, kd, vd, o, lse, causal=causal, cu_seqlens=cu)
    dq, dk, dv = (torch.full_like(x, float("nan")) for x in (qd, kd, vd))
    uly.ulysses_attn_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, causal=causal, cu_seqlens=cu)
    torch.cuda.synchronize()
    assert uly.ulysses_get_device_status()[0] == 0
    dq_r, dk_r, dv_r, o_r, lse_r = oracle.attn_bwd(q, k, v, do, causal=causal, cu_seqlens=cu)
    # with one token dS = dP - D vanishes: dQ and dK are exactly 0, so their
    # error is measured against the size of the other gradients instead
    floor = float(np.linalg.norm(dv_r)) if N == 1 else 1e-300
    errs = dict(o=rel_fro(o, o_r), dq=rel_fro(dq, dq_r, floor), dk=rel_fro(dk, dk_r, floor),
                dv=rel_fro(dv, dv_r))
    lse_err = max_abs(lse, lse_r)
    log_errors(f"attn S{S} B{B} N{N} Hq{Hq} Hkv{Hkv} d{d} {tag} causal{int(causal)} docs{0 if cu is None else len(cu) - 1}",
               lse_max_abs=lse_err, **errs)
    for name, e in errs.items():
        assert e <= REL_TOL[tag], (name, e, errs, lse_err)
    assert lse_err <= LSE_TOL[tag], (lse_err, errs)
    return errs, lse_err


BF16_CASES = [
    # S, B, N, Hq, Hkv, causal, cu
    (2, 1, 300, 4, 2, True, None),            # ragged tail, two shards
    (1, 2, 512, 8, 2, True, None),            # GQA group of 4, two batches
    (1, 1, 257, 3, 1, True, None),            # odd group: one head has no partner
    (1, 1, 200, 2, 2, False, None),           # non-causal, no GQA
    (1, 1, 700, 4, 1, True, [0, 100, 101, 350, 700]),   # packed docs, 1-token doc
    (1, 1, 450, 2, 1, False, [0, 129, 300, 450]),       # block-diagonal, non-causal
    (1, 1, 1, 2, 1, True, None),              # a single token
    (1, 1, 640, 2, 2, True, None),            # exact multiple of the tile
]


@pytest.mark.parametrize("S,B,N,Hq,Hkv,causal,cu", BF16_CASES)
def test_bf16_attention_vs_oracle(uly, S, B, N, Hq, Hkv, causal, cu):
    _attn_case(uly, S, B, N, Hq, Hkv, 128, torch.bfloat16, causal, cu)


FP32_CASES = [
    (2, 1, 130, 4, 4, 64, True, None),
    (1, 2, 77, 4, 2, 128, True, None),
    (1, 1, 90, 2, 1, 64, False, [0, 1, 40, 90]),
    (1, 1, 1, 1, 1, 64, True, None),
]


@pytest.mark.parametrize("S,B,N,Hq,Hkv,d,causal,cu", FP32_CASES)
def test_fp32_attention_vs_oracle(uly, S, B, N, Hq, Hkv, d, causal, cu):
    _attn_case(uly, S, B, N, Hq, Hkv, d, torch.float32, causal, cu)


def test_one_token_documents_copy_values(uly):
    """Every document of length 1: each row attends only to itself, o_i = v_i."""
    N, Hq, Hkv = 256, 2, 1
    cu = list(range(N + 1))
    q = _rand((1, 1, N, Hq, 128), 7, torch.bfloat16).cuda()
    k = _rand((1, 1, N, Hkv, 128), 8, torch.bfloat16).cuda()
    v = _rand((1, 1, N, Hkv, 128), 9, torch.bfloat16).cuda()
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, Hq, N, dtype=torch.float32, device="cuda")
    uly.ulysses_attn_fwd(q, k, v, o, lse, causal=True, cu_seqlens=cu)
    torch.cuda.synchronize()
    for h in range(Hq):
        assert torch.equal(o[0, 0, :, h], v[0, 0, :, 0])


def test_tiny_fp32_workload_full_path(uly, oracle_mod):
    """The fp32 N=256, P=2 workload through every step, against the oracle."""
    w = WORKLOADS["tiny_fp32_n256"]
    seq = draw_seq_inputs(w, seed=0)
    out = run_path(uly, seq, w.P)
    oh = {n: oracle_mod.seq_to_head(seq[n], w.P) for n in ("q", "k", "v", "dout")}
    for n in ("q", "k", "v", "dout"):
        assert bytes_equal(out[n + "_h"], oh[n])
    dq, dk, dv, o, lse = oracle_mod.attn_bwd(oh["q"], oh["k"], oh["v"], oh["dout"])
    assert rel_fro(out["o_h"], o) <= REL_TOL["fp32"]
    assert max_abs(out["lse"], lse) <= LSE_TOL["fp32"]
    for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert rel_fro(out[name + "_h"], ref) <= REL_TOL["fp32"], name
    # back in the sequence layout
    o_seq = oracle_mod.head_to_seq(torch.from_numpy(o), w.P)
    assert rel_fro(out["o_seq"], o_seq) <= REL_TOL["fp32"]
    dq_seq = oracle_mod.head_to_seq(torch.from_numpy(dq), w.P)
    assert rel_fro(out["dq_seq"], dq_seq) <= REL_TOL["fp32"]


def test_small_bf16_ulysses_path(uly, oracle_mod):
    """Qwen3-4B head shapes at N=1024, P=4: the whole bf16 path vs the oracle."""
    w = WORKLOADS["qwen3_4b_n8192"]
    seq = draw_seq_inputs(w, seed=5, N=1024)
    out = run_path(uly, seq, w.P)
    oh = {n: oracle_mod.seq_to_head(seq[n], w.P) for n in ("q", "k", "v", "dout")}
    for n in oh:
        assert bytes_equal(out[n + "_h"], oh[n])
    dq, dk, dv, o, lse = oracle_mod.attn_bwd(oh["q"], oh["k"], oh["v"], oh["dout"])
    for name, ref in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        ref_seq = oracle_mod.head_to_seq(torch.from_numpy(ref), w.P)
        assert rel_fro(out[name + "_seq"], ref_seq) <= REL_TOL["bf16"], name
    assert max_abs(out["lse"], lse) <= LSE_TOL["bf16"]


def test_wait_timeout_reports_status(uly):
    """A wait on a flag nothing sets gives up, reports ULY_ERR_TIMEOUT with its
    site, and the context stays usable."""
    uly.ulysses_selftest_wait_timeout(2_000_000)  # 2 ms
    st, site = uly.ulysses_get_device_status()
    assert st == 6 and site == 0x7E
    assert uly.ulysses_get_device_status()[0] == 0  # cleared
    x = torch.arange(16, dtype=torch.float32, device="cuda")
    assert float(x.sum()) == 120.0
