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
    g = Guards()
    for name, x, H in (("q", q, Hq), ("k", k, Hkv), ("v", v, Hkv), ("dout", do, Hq)):
        h = g.empty((P, B, N, H // P, d), x.dtype)
        uly.ulysses_seq_to_head(x, h, P)
        out[name + "_h"] = h
    S = P if attn_shards is None else attn_shards
    qh, kh, vh, doh = (out[n][:S] for n in ("q_h", "k_h", "v_h", "dout_h"))
    o = g.empty(qh.shape, qh.dtype)
    lse = g.empty((S, B, Hq // P, N), torch.float32)
    uly.ulysses_attn_fwd(qh, kh, vh, o, lse, causal=causal, cu_seqlens=cu)
    dq, dk, dv = g.empty(qh.shape, qh.dtype), g.empty(kh.shape, kh.dtype), g.empty(vh.shape, vh.dtype)
    uly.ulysses_attn_bwd(qh, kh, vh, o, lse, doh, dq, dk, dv, causal=causal, cu_seqlens=cu)
    out.update(o_h=o, lse=lse, dq_h=dq, dk_h=dk, dv_h=dv)
    if S == P:
        for name, x, H in (("o", o, Hq), ("dq", dq, Hq), ("dk", dk, Hkv), ("dv", dv, Hkv)):
            s_ = g.empty((P, B, N // P, H, d), x.dtype)
            uly.ulysses_head_to_seq(x, s_, P)
            out[name + "_seq"] = s_
    torch.cuda.synchronize()
    st, site = uly.ulysses_get_device_status()
    assert st == 0, f"device status {st} at site {site:#x}"
    g.check()
    return out


class Guards:
    """Device buffers fenced by sentinel bytes.

    Each buffer handed out sits inside a larger allocation with PAD bytes of a
    fixed pattern before and after it.  A kernel that writes past either end
    of an output (a ragged tail, a padded row, an index off by one tile)
    changes a sentinel, which ``check()`` reports; NaN-prefilled outputs only
    catch elements that were never written.  The views are contiguous, keep
    the allocation's 16-byte alignment and can be passed wherever a plain
    tensor is expected."""
    PAD = 4096
    SENTINEL = 0xA5

    def __init__(self, device="cuda"):
        self.device = device
        self._bufs = []

    def empty(self, shape, dtype, fill=None):
        shape = tuple(int(s) for s in shape)
        esize = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) * esize
        raw = torch.full((self.PAD + n + self.PAD,), self.SENTINEL, dtype=torch.uint8, device=self.device)
        view = raw[self.PAD:self.PAD + n].view(dtype).view(shape)
        if fill is not None:
            view.fill_(fill)
        self._bufs.append((raw, n, shape))
        return view

    def full_like(self, x, fill):
        return self.empty(x.shape, x.dtype, fill)

    def workspace(self, nbytes):
        return self.empty((max(int(nbytes), 256),), torch.uint8)

    def check(self):
        torch.cuda.synchronize()
        for raw, n, shape in self._bufs:
            head = raw[:self.PAD]
            tail = raw[self.PAD + n:]
            bad_head = int((head != self.SENTINEL).sum())
            bad_tail = int((tail != self.SENTINEL).sum())
            assert bad_head == 0 and bad_tail == 0, (
                f"write outside a buffer of shape {shape}: {bad_head} bytes changed before it, "
                f"{bad_tail} after it")
