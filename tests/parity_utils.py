"""Helpers shared by the GPU parity tests: error metrics, tolerances and a
driver that runs the whole Ulysses path through the C ABI.

Tolerances (attention outputs O, dQ, dK, dV): relative Frobenius error
<= 5e-3 for bf16 and <= 1e-5 for fp32; the log-sum-exp: max abs error
<= 2e-3 (bf16) / 1e-5 (fp32).  Swaps: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

REL_TOL = {"bf16": 5e-3, "fp32": 1e-5}
LSE_TOL = {"bf16": 2e-3, "fp32": 1e-5}


def to64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def rel_fro(gpu, ref, floor: float = 1e-300) -> float:
    """||gpu - ref||_F / max(||ref||_F, floor).  A floor is needed where the
    exact result vanishes (e.g. dQ and dK of a one-token sequence)."""
    g, r = to64(gpu), to64(ref)
    return float(np.linalg.norm((g - r).ravel()) / max(np.linalg.norm(r.ravel()), floor))


def log_errors(case: str, **errs) -> None:
    """Append measured errors to $PARITY_LOG (JSON lines) when it is set."""
    import json
    import os
    path = os.environ.get("PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": case, **{k: float(v) for k, v in errs.items()}}) + "\n")


def max_abs(gpu, ref) -> float:
    return float(np.max(np.abs(to64(gpu) - to64(ref))))


def bytes_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    a = a.detach().contiguous().cpu()
    b = b.detach().contiguous().cpu()
    return a.shape == b.shape and torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def run_path(uly, seq: dict, P: int, causal: bool = True, cu=None, attn_shards=None):
    """seq->head, attention fwd, head->seq; dO seq->head, attention bwd,
    dQ/dK/dV head->seq.  All on the GPU through the C ABI; returns a dict of
    device tensors."""
    q, k, v, do = (seq[n].cuda().contiguous() for n in ("q", "k", "v", "dout"))
    Ps, B, Np, Hq, d = q.shape
    Hkv = k.shape[3]
    N = Np * P
    out = {}
    for name, x, H in (("q", q, Hq), ("k", k, Hkv), ("v", v, Hkv), ("dout", do, Hq)):
        h = torch.empty(P, B, N, H // P, d, dtype=x.dtype, device="cuda")
        uly.ulysses_seq_to_head(x, h, P)
        out[name + "_h"] = h
    S = P if attn_shards is None else attn_shards
    qh, kh, vh, doh = (out[n][:S] for n in ("q_h", "k_h", "v_h", "dout_h"))
    o = torch.empty_like(qh)
    lse = torch.empty(S, B, Hq // P, N, dtype=torch.float32, device="cuda")
    uly.ulysses_attn_fwd(qh, kh, vh, o, lse, causal=causal, cu_seqlens=cu)
    dq, dk, dv = torch.empty_like(qh), torch.empty_like(kh), torch.empty_like(vh)
    uly.ulysses_attn_bwd(qh, kh, vh, o, lse, doh, dq, dk, dv, causal=causal, cu_seqlens=cu)
    out.update(o_h=o, lse=lse, dq_h=dq, dk_h=dk, dv_h=dv)
    if S == P:
        for name, x, H in (("o", o, Hq), ("dq", dq, Hq), ("dk", dk, Hkv), ("dv", dv, Hkv)):
            s_ = torch.empty(P, B, N // P, H, d, dtype=x.dtype, device="cuda")
            uly.ulysses_head_to_seq(x, s_, P)
            out[name + "_seq"] = s_
    torch.cuda.synchronize()
    st, site = uly.ulysses_get_device_status()
    assert st == 0, f"device status {st} at site {site:#x}"
    return out
