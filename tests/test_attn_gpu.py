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
from parity_utils import LSE_TOL, REL_TOL, Guards, bytes_equal, log_errors, max_abs, rel_fro, run_path
from ulysses_inputs import WORKLOADS, draw_seq_inputs

pytestmark = pytest.mark.gpu


def _rand(shape, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


def _attn_case(uly, S, B, N, Hq, Hkv, d, dtype, causal, cu, seed=0):
    q = _rand((S, B, N, Hq, d), seed + 1, dtype)
    k = _rand((S, B, N, Hkv, d), seed + 2, dtype)
    v = _rand((S, B, N, Hkv, d), seed + 3, dtype)
    do = _rand((S, B, N, Hq, d), seed + 4, dtype)
    return _attn_inputs_case(uly, q, k, v, do, causal, cu)


def _attn_inputs_case(uly, q, k, v, do, causal, cu, label="", tol=None):
    """Forward and backward on the GPU against the oracle for given inputs.
    `tol` overrides the relative bound of named outputs."""
    S, B, N, Hq, d = q.shape
    Hkv = k.shape[3]
    tag = "bf16" if q.dtype == torch.bfloat16 else "fp32"
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    g = Guards()
    nd = 0 if cu is None else len(cu) - 1
    o = g.full_like(qd, float("nan"))
    lse = g.empty((S, B, Hq, N), torch.float32, float("nan"))
    ws_f = g.workspace(uly.ulysses_attn_workspace_size(B, N, Hq, Hkv, d, S, nd, False, q.dtype))
    uly.ulysses_attn_fwd(qd, kd, vd, o, lse, causal=causal, cu_seqlens=cu, workspace=ws_f)
    g.check()
    dq, dk, dv = (g.full_like(x, float("nan")) for x in (qd, kd, vd))
    ws_b = g.workspace(uly.ulysses_attn_workspace_size(B, N, Hq, Hkv, d, S, nd, True, q.dtype))
    uly.ulysses_attn_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, causal=causal, cu_seqlens=cu, workspace=ws_b)
    torch.cuda.synchronize()
    assert uly.ulysses_get_device_status()[0] == 0
    g.check()
    dq_r, dk_r, dv_r, o_r, lse_r = oracle.attn_bwd(q, k, v, do, causal=causal, cu_seqlens=cu)
    # with one token dS = dP - D vanishes: dQ and dK are exactly 0, so their
    # error is measured against the size of the other gradients instead
    floor = float(np.linalg.norm(dv_r)) if N == 1 else 1e-300
    errs = dict(o=rel_fro(o, o_r), dq=rel_fro(dq, dq_r, floor), dk=rel_fro(dk, dk_r, floor),
                dv=rel_fro(dv, dv_r))
    lse_err = max_abs(lse, lse_r)
    log_errors(f"attn{label} S{S} B{B} N{N} Hq{Hq} Hkv{Hkv} d{d} {tag} causal{int(causal)} "
               f"docs{0 if cu is None else len(cu) - 1}", lse_max_abs=lse_err, **errs)
    for name, e in errs.items():
        bound = (tol or {}).get(name, REL_TOL[tag])
        assert e <= bound, (name, e, bound, errs, lse_err)
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
    (1, 1, 384, 8, 1, True, None),            # GQA group of 8: four head pairs share one KV head
    (1, 1, 600, 4, 2, True, [0, 0, 128, 128, 300, 600, 600]),  # zero-length documents at tile edges
    (2, 2, 384, 4, 2, True, [0, 200, 384]),   # documents with two shards and two batches
    (1, 1, 300, 3, 1, False, [0, 150, 300]),  # documents with an odd group (one head has no partner)
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


def _ramp_inputs(N, Hq, Hkv, d, seed, kind):
    """bf16 inputs whose scores move far along the key axis.  q_i ~ 8 u and
    k_j ~ a_j u (u a random unit vector) plus N(0, 1/4) noise, so
    s_ij ~ 8 a_j / sqrt(d):
      "rise":  a_j = 57 j / N, scores climb ~40 (natural log units) across the
               row, so the running maximum keeps jumping by more than the
               forward's 2^8 rescale threshold;
      "fall":  the mirror image, the first key tile holds the maximum;
      "spike": a_j = 0 except two late keys with scores ~40;
      "stairs": a_j constant over each 128-key tile, at levels (log2 units)
               0, 4, 14, 15, 19, 29, 30, 31: see test_running_max_speculation."""
    g = torch.Generator().manual_seed(seed)
    u = torch.randn(d, generator=g, dtype=torch.float64)
    u /= u.norm()
    t = torch.arange(N, dtype=torch.float64) / N
    if kind == "rise":
        a = 57.0 * t
    elif kind == "fall":
        a = 57.0 * (1.0 - t)
    elif kind == "stairs":
        levels = torch.tensor([0.0, 4.0, 14.0, 15.0, 19.0, 29.0, 30.0, 31.0], dtype=torch.float64)
        # s = 8 a / sqrt(d) natural-log units = level log2 units
        a = (levels * math.log(2.0) * math.sqrt(d) / 8.0).repeat_interleave(128)[:N]
    else:
        a = torch.zeros(N, dtype=torch.float64)
        a[int(0.7 * N)] = a[int(0.9 * N)] = 40.0 * math.sqrt(d) / 8.0
    q = 0.5 * torch.randn(1, 1, N, Hq, d, generator=g, dtype=torch.float64) + 8.0 * u
    k = 0.5 * torch.randn(1, 1, N, Hkv, d, generator=g, dtype=torch.float64) + a[None, None, :, None, None] * u
    v = torch.randn(1, 1, N, Hkv, d, generator=g, dtype=torch.float64)
    do = torch.randn(1, 1, N, Hq, d, generator=g, dtype=torch.float64)
    return [x.to(torch.bfloat16) for x in (q, k, v, do)]


def _dq_bf16_operand_error(q, k, v, do, causal):
    """Relative error of dQ computed exactly from the bf16-rounded operands
    the tensor cores must use: P rounded to bf16, dS = P (dP - D) rounded to
    bf16, dQ = scale dS K.  Since sum_j dS_ij = 0, dQ is what remains of a
    cancellation over the keys; when every k_j shares a large component the
    rounding of dS does not cancel and sets a floor on dQ's error no kernel
    with bf16 dS can go below."""
    S, B, N, Hq, d = q.shape
    G = Hq // k.shape[3]
    scale = 1.0 / math.sqrt(d)
    num = den = 0.0
    for h in range(Hq):
        qq, kk, vv, dd = (x[0, 0, :, hh].double() for x, hh in ((q, h), (k, h // G), (v, h // G), (do, h)))
        s_ = scale * (qq @ kk.T)
        if causal:
            s_ = s_.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -math.inf)
        p_ = torch.softmax(s_, dim=1)
        o_ = p_ @ vv
        dp = dd @ vv.T
        D = (dd * o_).sum(dim=1, keepdim=True)
        exact = scale * ((p_ * (dp - D)) @ kk)
        pb = p_.to(torch.bfloat16).double()
        dsb = (pb * (dp - D)).to(torch.bfloat16).double()
        emul = scale * (dsb @ kk)
        num += float(((emul - exact) ** 2).sum())
        den += float((exact ** 2).sum())
    return math.sqrt(num / den)


def _rescale_events(q, k, causal, tile=128):
    """How many times per row the running maximum of the scaled scores (log2
    units, over 128-key tiles in order) grows by more than 8: the rows on which
    the forward must rescale O held in TMEM."""
    d = q.shape[-1]
    qq = q[0, 0, :, 0].double()
    kk = k[0, 0, :, 0].double()
    s = (qq @ kk.T) * (1.0 / math.sqrt(d)) * (1.0 / math.log(2.0))
    N = s.shape[0]
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -math.inf)
    tmax = torch.stack([s[:, c:c + tile].max(dim=1).values for c in range(0, N, tile)], dim=1)
    events = torch.zeros(N, dtype=torch.int64)
    m = tmax[:, 0].clone()
    for c in range(1, tmax.shape[1]):
        jump = tmax[:, c] > m + 8.0
        events += jump.long()
        m = torch.where(jump, tmax[:, c], m)
    return events


@pytest.mark.parametrize("kind", ["rise", "fall", "spike"])
@pytest.mark.parametrize("causal", [True, False])
def test_score_ramps_exercise_the_rescale(uly, kind, causal):
    """Scores that climb, fall or jump along the key axis: the lazy O rescale
    in the forward (and the backward's use of the resulting lse) against the
    oracle.  The rising and spiking inputs are checked to cross the rescale
    threshold on most rows."""
    N, Hq, Hkv, d = 1024, 4, 2, 128
    q, k, v, do = _ramp_inputs(N, Hq, Hkv, d, seed=31, kind=kind)
    ev = _rescale_events(q, k, causal)
    if kind == "rise":
        assert float((ev[N // 2:] >= 2).double().mean()) > 0.9, ev[N // 2:].float().mean()
    if kind == "spike":
        assert float((ev[int(0.9 * N):] >= 1).double().mean()) > 0.9
    if kind == "fall" and causal:
        assert int(ev.sum()) == 0
    # O, lse, dK, dV: the plain bf16 bounds.  dQ: within twice the error that
    # exact arithmetic on the bf16-rounded P and dS already has (never looser
    # than the plain bound) -- see _dq_bf16_operand_error.
    floor = _dq_bf16_operand_error(q, k, v, do, causal)
    _attn_inputs_case(uly, q, k, v, do, causal, None, label=f" ramp-{kind}",
                      tol={"dq": max(REL_TOL["bf16"], 2.0 * floor)})


def _speculation_paths(q, k, causal, tile=128):
    """Per (row, key tile) after a row's first tile, which way the forward's
    running-maximum speculation goes (query head 0, log2 units): "kept" when
    the tile's exponentials against the running maximum m sum to at most 2^8;
    otherwise the tile is redone exactly, "grow" if its maximum exceeds m + 8
    (m moves, O is rescaled) and "redo" if not (m stays)."""
    d = q.shape[-1]
    s = (q[0, 0, :, 0].double() @ k[0, 0, :, 0].double().T) * (1.0 / math.sqrt(d)) / math.log(2.0)
    N = s.shape[0]
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -math.inf)
    counts = {"kept": 0, "redo": 0, "grow": 0}
    for i in range(N):
        m = -math.inf
        for c in range(0, N, tile):
            x = s[i, c:c + tile]
            mx = float(x.max())
            if mx == -math.inf and m == -math.inf:
                continue
            if m == -math.inf:
                m = mx
            elif float(torch.exp2(x - m).sum()) <= 256.0:
                counts["kept"] += 1
            elif mx > m + 8.0:
                counts["grow"] += 1
                m = mx
            else:
                counts["redo"] += 1
    return counts


@pytest.mark.parametrize("causal", [True, False])
def test_running_max_speculation(uly, causal):
    """Key tiles at stepped score levels drive every branch of the forward's
    speculative running maximum: tiles kept on the speculation, tiles redone
    with the maximum unchanged (their exponentials sum above 2^8 while none
    lies more than 8 above the running maximum in log2 units) and tiles where
    the maximum moves and O is rescaled.  Results against the oracle."""
    N, Hq, Hkv, d = 1024, 4, 2, 128
    q, k, v, do = _ramp_inputs(N, Hq, Hkv, d, seed=37, kind="stairs")
    paths = _speculation_paths(q, k, causal)
    assert all(n >= 100 for n in paths.values()), paths
    floor = _dq_bf16_operand_error(q, k, v, do, causal)
    _attn_inputs_case(uly, q, k, v, do, causal, None, label=" stairs",
                      tol={"dq": max(REL_TOL["bf16"], 2.0 * floor)})


@pytest.mark.parametrize("causal", [True, False])
def test_one_document_matches_no_documents(uly, causal):
    """cu_seqlens = [0, N] describes the same mask as no documents, but runs
    the kernel instances built for packed documents (tiles in the host's
    walk order; in the forward a row's first tile from registers).  Each
    unit computes the same thing in both, so O, lse, dK and dV must agree
    bit for bit; dQ only up to the order of its fp32 reductions."""
    S, N, Hq, Hkv = 2, 1000, 8, 2  # ragged tail, GQA groups of 4 (two head pairs)
    q = _rand((S, 1, N, Hq, 128), 21, torch.bfloat16).cuda()
    k = _rand((S, 1, N, Hkv, 128), 22, torch.bfloat16).cuda()
    v = _rand((S, 1, N, Hkv, 128), 23, torch.bfloat16).cuda()
    do = _rand((S, 1, N, Hq, 128), 24, torch.bfloat16).cuda()
    out = {}
    for name, cu in (("none", None), ("one", [0, N])):
        g = Guards()
        nd = 0 if cu is None else 1
        o = g.full_like(q, float("nan"))
        lse = g.empty((S, 1, Hq, N), torch.float32, float("nan"))
        ws_f = g.workspace(uly.ulysses_attn_workspace_size(1, N, Hq, Hkv, 128, S, nd, False, torch.bfloat16))
        uly.ulysses_attn_fwd(q, k, v, o, lse, causal=causal, cu_seqlens=cu, workspace=ws_f)
        dq, dk, dv = (g.full_like(x, float("nan")) for x in (q, k, v))
        ws_b = g.workspace(uly.ulysses_attn_workspace_size(1, N, Hq, Hkv, 128, S, nd, True, torch.bfloat16))
        uly.ulysses_attn_bwd(q, k, v, o, lse, do, dq, dk, dv, causal=causal, cu_seqlens=cu, workspace=ws_b)
        torch.cuda.synchronize()
        assert uly.ulysses_get_device_status()[0] == 0
        g.check()
        out[name] = (o, lse, dq, dk, dv)
    (o0, l0, dq0, dk0, dv0), (o1, l1, dq1, dk1, dv1) = out["none"], out["one"]
    for a, b, what in ((o0, o1, "o"), (l0, l1, "lse"), (dk0, dk1, "dk"), (dv0, dv1, "dv")):
        assert bytes_equal(a, b), what
    assert rel_fro(dq1, dq0) <= 1e-3, rel_fro(dq1, dq0)


def test_one_token_documents_copy_values(uly):
    """Every document of length 1: each row attends only to itself, o_i = v_i."""
    N, Hq, Hkv = 256, 2, 1
    cu = list(range(N + 1))
    q = _rand((1, 1, N, Hq, 128), 7, torch.bfloat16).cuda()
    k = _rand((1, 1, N, Hkv, 128), 8, torch.bfloat16).cuda()
    v = _rand((1, 1, N, Hkv, 128), 9, torch.bfloat16).cuda()
    g = Guards()
    o = g.empty(q.shape, q.dtype)
    lse = g.empty((1, 1, Hq, N), torch.float32)
    uly.ulysses_attn_fwd(q, k, v, o, lse, causal=True, cu_seqlens=cu)
    torch.cuda.synchronize()
    g.check()
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


def _random_cases(n, seed=1234):
    """Seeded random shapes: shards, batches, ragged lengths, GQA groups of
    1-8, causal or not, and documents (none, or lengths >= 8 with a
    zero-length document sometimes in between)."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        S, B = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        N = int(rng.integers(2, 700))
        Hkv = int(rng.integers(1, 3))
        G = int(rng.choice([1, 2, 3, 4, 8]))
        causal = bool(rng.integers(0, 2))
        cu = None
        if i % 2 == 1 and N >= 16:  # every other case packs documents
            cu, t = [0], 0
            while t < N:
                L = min(int(rng.integers(8, max(9, N // 2))), N - t)
                t += L
                cu.append(t)
                if rng.integers(0, 4) == 0:
                    cu.append(t)  # a zero-length document
            if N - (cu[-1] - cu[-2]) > 0 and cu[-1] - cu[-2] < 8 and len(cu) > 2:
                cu.pop(-2)  # keep the last real document at least 8 long
        cases.append((S, B, N, G * Hkv, Hkv, causal, cu))
    return cases


@pytest.mark.parametrize("S,B,N,Hq,Hkv,causal,cu", _random_cases(12))
def test_random_shapes_vs_oracle(uly, S, B, N, Hq, Hkv, causal, cu):
    _attn_case(uly, S, B, N, Hq, Hkv, 128, torch.bfloat16, causal, cu, seed=5)
