"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (all P head shards in one call; one shard for the 1M case).

The oracle cannot afford full quadratic attention here, so it checks what it
can compute one by one -- sampled query rows of O, lse and dQ, sampled key
rows of dK and dV (keys near the end of a document, which few rows attend)
-- and the swaps bit for bit in full.  Properties that hold at any size are
checked on every output: sum_j dV_j equals the group sum of sum_i dO_i, and
sum_j dK_j = 0.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_utils import LSE_TOL, REL_TOL, bytes_equal, log_errors, rel_fro, to64
from ulysses_inputs import WORKLOADS, cu_seqlens_from_lengths, doc_lengths, draw_seq_inputs

pytestmark = pytest.mark.gpu


def _pipeline(uly, w, seed, cu):
    dev = "cuda" if w.N >= 65536 else "cpu"
    seq = draw_seq_inputs(w, seed=seed, device=dev)
    P, S = w.P, w.shards_timed
    out = {"seq": seq}
    heads = {}
    for name, H in (("q", w.Hq), ("k", w.Hkv), ("v", w.Hkv), ("dout", w.Hq)):
        x = seq[name].cuda()
        h = torch.empty(P, w.B, w.N, H // P, w.d, dtype=x.dtype, device="cuda")
        uly.ulysses_seq_to_head(x, h, P)
        heads[name] = h
    qh, kh, vh, doh = (heads[n][:S] for n in ("q", "k", "v", "dout"))
    o = torch.empty_like(qh)
    lse = torch.empty(S, w.B, w.Hp, w.N, dtype=torch.float32, device="cuda")
    uly.ulysses_attn_fwd(qh, kh, vh, o, lse, causal=True, cu_seqlens=cu)
    dq, dk, dv = torch.empty_like(qh), torch.empty_like(kh), torch.empty_like(vh)
    uly.ulysses_attn_bwd(qh, kh, vh, o, lse, doh, dq, dk, dv, causal=True, cu_seqlens=cu)
    torch.cuda.synchronize()
    assert uly.ulysses_get_device_status()[0] == 0
    out.update(heads=heads, o=o, lse=lse, dq=dq, dk=dk, dv=dv, S=S)
    return out


def _doc_end(cu, j):
    k = int(np.searchsorted(cu, j, side="right")) - 1
    return int(cu[k + 1])


@pytest.mark.parametrize("name,n_rows,n_keys", [
    ("qwen3_4b_n8192", 96, 8),
    ("packed_docs_n32768", 96, 8),
    ("qwen3_4b_n65536", 64, 6),
    ("single_shard_n1m", 256, 3),
])
def test_full_size_sampled(uly, oracle_mod, name, n_rows, n_keys):
    w = WORKLOADS[name]
    cu = None
    if w.packed_docs:
        cu = cu_seqlens_from_lengths(doc_lengths(w.N, w.P, seed=3))
    r = _pipeline(uly, w, seed=3, cu=cu)
    S = r["S"]
    # the oracle's own swap of the same inputs, checked bit for bit in full
    oh = {}
    for n in ("q", "k", "v", "dout"):
        ref = oracle_mod.seq_to_head(r["seq"][n].cpu(), w.P)
        assert bytes_equal(r["heads"][n], ref), n
        oh[n] = ref[:S]
    del r["heads"]
    rng = np.random.default_rng(11)
    rows = [(int(rng.integers(S)), 0, int(rng.integers(w.Hp)), int(i))
            for i in np.concatenate([rng.integers(0, w.N, n_rows - 4), [0, 1, w.N - 2, w.N - 1]])]
    o_ref, lse_ref = oracle_mod.attn_fwd_rows(oh["q"], oh["k"], oh["v"], rows, cu_seqlens=cu)
    o_gpu = np.stack([to64(r["o"][s, b, i, h]) for s, b, h, i in rows])
    lse_gpu = np.array([float(r["lse"][s, b, h, i]) for s, b, h, i in rows])
    assert rel_fro(o_gpu, o_ref) <= REL_TOL["bf16"]
    assert np.max(np.abs(lse_gpu - lse_ref)) <= LSE_TOL["bf16"]
    qrows = rows[: max(8, n_rows // 4)]
    dq_ref = oracle_mod.attn_bwd_q_rows(oh["q"], oh["k"], oh["v"], oh["dout"], qrows, cu_seqlens=cu)
    dq_gpu = np.stack([to64(r["dq"][s, b, i, h]) for s, b, h, i in qrows])
    assert rel_fro(dq_gpu, dq_ref) <= REL_TOL["bf16"]
    # key rows near the end of their document: few rows attend to them
    ends = [w.N] if cu is None else [int(c) for c in cu[1:]]
    keys = []
    for t in range(n_keys):
        e = ends[int(rng.integers(len(ends)))]
        j = e - 1 - int(rng.integers(0, 24))
        keys.append((int(rng.integers(S)), 0, int(rng.integers(w.Hkvp)), max(j, 0)))
    dk_ref, dv_ref = oracle_mod.attn_bwd_kv_rows(oh["q"], oh["k"], oh["v"], oh["dout"], keys, cu_seqlens=cu)
    dk_gpu = np.stack([to64(r["dk"][s, b, j, h]) for s, b, h, j in keys])
    dv_gpu = np.stack([to64(r["dv"][s, b, j, h]) for s, b, h, j in keys])
    errs = dict(o=rel_fro(o_gpu, o_ref), lse_max_abs=float(np.max(np.abs(lse_gpu - lse_ref))),
                dq=rel_fro(dq_gpu, dq_ref), dk=rel_fro(dk_gpu, dk_ref), dv=rel_fro(dv_gpu, dv_ref))
    log_errors(f"{name} sampled rows={len(rows)} dq_rows={len(qrows)} kv_rows={len(keys)}", **errs)
    assert errs["dk"] <= REL_TOL["bf16"], errs
    assert errs["dv"] <= REL_TOL["bf16"], errs
    # invariants on every output (fp64 sums of the bf16 results)
    G = w.G
    dv_sum = r["dv"].double().sum(dim=2)                       # [S][B][Hkvp][d]
    do_h = oh["dout"].double().sum(dim=2)                      # [S][B][Hp][d]
    do_grp = do_h.view(S, w.B, w.Hkvp, G, w.d).sum(dim=3)
    err = (dv_sum.cpu() - do_grp).norm() / do_grp.norm()
    assert float(err) <= 5e-3, float(err)
    dk_sum = r["dk"].double().sum(dim=2).cpu()                 # should vanish
    scale_ref = r["dk"].double().abs().sum(dim=2).cpu()
    assert float(dk_sum.abs().max() / scale_ref.max()) <= 5e-3
