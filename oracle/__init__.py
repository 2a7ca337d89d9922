"""fp64 CPU oracle for the Ulysses swap + attention path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by ``bench.py``'s CPU-baseline leg, never by the product package.  It shares
no code with the CUDA library.

``oracle.c`` holds the swap index maps and the attention definitions (see its
header).  This module compiles it with gcc (``build()``), wraps it with ctypes
and adds the loss aggregation (``loss.py``).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, a library cross-check, finite differences, the Ulysses
diagram); see the individual test docstrings.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np
import torch

from .loss import (aggregate_sharded_loss, aggregated_loss_grad,  # noqa: F401
                   full_sequence_loss, per_rank_losses, per_rank_losses_batched, shift_labels,
                   shift_labels_batched)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.oracle_num_threads.restype = i32
            for name in ("oracle_seq_to_head", "oracle_head_to_seq"):
                f = getattr(lib, name)
                f.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64]
                f.restype = None
            shape = [i64, i64, i64, i64, i64, i64, i32, vp, i32, dbl]
            lib.oracle_attn_fwd.argtypes = [vp] * 5 + shape
            lib.oracle_attn_fwd_rows.argtypes = [vp] * 3 + shape + [vp, i64, vp, vp]
            lib.oracle_attn_bwd.argtypes = [vp] * 9 + shape
            lib.oracle_attn_bwd_q_rows.argtypes = [vp] * 4 + shape + [vp, i64, vp]
            lib.oracle_attn_bwd_kv_rows.argtypes = [vp] * 4 + shape + [vp, i64, vp, vp]
            for name in ("oracle_attn_fwd", "oracle_attn_fwd_rows", "oracle_attn_bwd",
                         "oracle_attn_bwd_q_rows", "oracle_attn_bwd_kv_rows"):
                getattr(lib, name).restype = None
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _f64(x) -> np.ndarray:
    """Exact upcast of a torch tensor (bf16/fp32/fp64) or array to fp64."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().to(torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _bytes(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        t = x.detach().contiguous().cpu()
        return np.ascontiguousarray(t.view(torch.uint8).reshape(-1).numpy())
    return np.ascontiguousarray(np.asarray(x)).view(np.uint8).reshape(-1)


# ------------------------------------------------------------------ swap

def seq_to_head(x_seq: torch.Tensor, P: int) -> torch.Tensor:
    """[P][B][N/P][H][d] -> [P][B][N][H/P][d], any dtype, byte copy."""
    Pp, B, Np, H, d = x_seq.shape
    assert Pp == P and H % P == 0
    N = Np * P
    src = _bytes(x_seq)
    dst = np.empty_like(src)
    _load().oracle_seq_to_head(_ptr(src), _ptr(dst), B, N, H, d, P, x_seq.element_size())
    out = torch.from_numpy(dst).view(x_seq.dtype)
    return out.reshape(P, B, N, H // P, d)


def head_to_seq(x_head: torch.Tensor, P: int) -> torch.Tensor:
    """[P][B][N][H/P][d] -> [P][B][N/P][H][d], any dtype, byte copy."""
    Pp, B, N, Hp, d = x_head.shape
    assert Pp == P and N % P == 0
    H = Hp * P
    src = _bytes(x_head)
    dst = np.empty_like(src)
    _load().oracle_head_to_seq(_ptr(src), _ptr(dst), B, N, H, d, P, x_head.element_size())
    out = torch.from_numpy(dst).view(x_head.dtype)
    return out.reshape(P, B, N // P, H, d)


# ------------------------------------------------------------- attention

def _cu(cu_seqlens) -> tuple:
    if cu_seqlens is None:
        return None, 0
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    return cu, len(cu) - 1


def _scale(scale: Optional[float], d: int) -> float:
    return float(scale) if scale is not None and scale > 0 else 1.0 / float(np.sqrt(d))


def attn_fwd(q, k, v, causal: bool = True, cu_seqlens=None, scale: Optional[float] = None):
    """Attention forward over head shards.

    q [S][B][N][Hq][d], k/v [S][B][N][Hkv][d] (any float dtype; upcast exactly).
    Returns (o fp64 like q, lse fp64 [S][B][Hq][N]).
    """
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    S, B, N, Hq, d = q64.shape
    Hkv = k64.shape[3]
    cu, nd = _cu(cu_seqlens)
    o = np.empty_like(q64)
    lse = np.empty((S, B, Hq, N), dtype=np.float64)
    _load().oracle_attn_fwd(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(o), _ptr(lse),
                            S, B, N, Hq, Hkv, d, int(causal),
                            _ptr(cu) if cu is not None else None, nd, _scale(scale, d))
    return o, lse


def attn_fwd_rows(q, k, v, rows: Sequence[Sequence[int]], causal: bool = True,
                  cu_seqlens=None, scale: Optional[float] = None):
    """Sampled forward rows; rows = [(s, b, h, i), ...].  Returns (o [n][d], lse [n])."""
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    S, B, N, Hq, d = q64.shape
    Hkv = k64.shape[3]
    cu, nd = _cu(cu_seqlens)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 4))
    o = np.empty((len(r), d), dtype=np.float64)
    lse = np.empty((len(r),), dtype=np.float64)
    _load().oracle_attn_fwd_rows(_ptr(q64), _ptr(k64), _ptr(v64),
                                 S, B, N, Hq, Hkv, d, int(causal),
                                 _ptr(cu) if cu is not None else None, nd, _scale(scale, d),
                                 _ptr(r), len(r), _ptr(o), _ptr(lse))
    return o, lse


def attn_bwd(q, k, v, dout, causal: bool = True, cu_seqlens=None,
             scale: Optional[float] = None):
    """Full backward.  Returns (dq, dk, dv, o, lse), all fp64."""
    q64, k64, v64, do64 = _f64(q), _f64(k), _f64(v), _f64(dout)
    S, B, N, Hq, d = q64.shape
    Hkv = k64.shape[3]
    cu, nd = _cu(cu_seqlens)
    dq = np.empty_like(q64)
    dk = np.empty_like(k64)
    dv = np.empty_like(v64)
    o = np.empty_like(q64)
    lse = np.empty((S, B, Hq, N), dtype=np.float64)
    _load().oracle_attn_bwd(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(do64),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(o), _ptr(lse),
                            S, B, N, Hq, Hkv, d, int(causal),
                            _ptr(cu) if cu is not None else None, nd, _scale(scale, d))
    return dq, dk, dv, o, lse


def attn_bwd_q_rows(q, k, v, dout, rows, causal: bool = True, cu_seqlens=None,
                    scale: Optional[float] = None):
    """Sampled dq rows; rows = [(s, b, h, i), ...].  Returns dq [n][d]."""
    q64, k64, v64, do64 = _f64(q), _f64(k), _f64(v), _f64(dout)
    S, B, N, Hq, d = q64.shape
    Hkv = k64.shape[3]
    cu, nd = _cu(cu_seqlens)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 4))
    dq = np.empty((len(r), d), dtype=np.float64)
    _load().oracle_attn_bwd_q_rows(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(do64),
                                   S, B, N, Hq, Hkv, d, int(causal),
                                   _ptr(cu) if cu is not None else None, nd, _scale(scale, d),
                                   _ptr(r), len(r), _ptr(dq))
    return dq


def attn_bwd_kv_rows(q, k, v, dout, keys, causal: bool = True, cu_seqlens=None,
                     scale: Optional[float] = None):
    """Sampled dk/dv rows; keys = [(s, b, kvh, j), ...].  Returns (dk, dv) [n][d]."""
    q64, k64, v64, do64 = _f64(q), _f64(k), _f64(v), _f64(dout)
    S, B, N, Hq, d = q64.shape
    Hkv = k64.shape[3]
    cu, nd = _cu(cu_seqlens)
    r = np.ascontiguousarray(np.asarray(keys, dtype=np.int64).reshape(-1, 4))
    dk = np.empty((len(r), d), dtype=np.float64)
    dv = np.empty((len(r), d), dtype=np.float64)
    _load().oracle_attn_bwd_kv_rows(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(do64),
                                    S, B, N, Hq, Hkv, d, int(causal),
                                    _ptr(cu) if cu is not None else None, nd, _scale(scale, d),
                                    _ptr(r), len(r), _ptr(dk), _ptr(dv))
    return dk, dv
