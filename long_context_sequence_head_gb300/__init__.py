"""Python binding of the GB300 Ulysses library (``include/ulysses.h``).

Argument marshalling only: every step of the path (the seq<->head swaps, the
attention forward and backward) runs in the CUDA kernels of
``_build/libulysses_gb300.so``.  PyTorch provides device memory and streams.
There is no CPU fallback: if the library is missing, importing the functions
raises, and every call checks the status the C ABI returns.

The functions keep the C names.  Tensors must be contiguous CUDA tensors in
the layouts of the header:
    seq layout  [P][B][N/P][H][d]     head layout [P][B][N][H/P][d]
    q, o, dout  [S][B][N][Hq][d]      k, v        [S][B][N][Hkv][d]
    lse         [S][B][Hq][N] fp32
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

from . import build as _build_mod

ULY_OK = 0
ULY_BF16 = 0
ULY_FP32 = 1
_STATUS = {0: "ULY_OK", 1: "ULY_ERR_INVALID_ARG", 2: "ULY_ERR_UNSUPPORTED", 3: "ULY_ERR_MISALIGNED",
           4: "ULY_ERR_OVERLAP", 5: "ULY_ERR_CUDA", 6: "ULY_ERR_TIMEOUT", 7: "ULY_ERR_WORKSPACE",
           8: "ULY_ERR_SCRATCH_LIMIT", 9: "ULY_ERR_BOUNDS"}

# every symbol include/ulysses.h declares
EXPORTED = ("ulysses_seq_to_head", "ulysses_head_to_seq", "ulysses_swap_batch", "ulysses_attn_workspace_size",
            "ulysses_attn_tile_order",
            "ulysses_attn_fwd", "ulysses_attn_bwd", "ulysses_attn_fwd_seq", "ulysses_attn_bwd_seq",
            "ulysses_attn_bwd_noalloc", "ulysses_sharded_ce_workspace_size", "ulysses_sharded_ce_loss",
            "ulysses_ring_attn_workspace_size", "ulysses_ring_attn_fwd", "ulysses_ring_attn_bwd",
            "ulysses_get_device_status",
            "ulysses_set_wait_limit_ns", "ulysses_selftest_wait_timeout", "ulysses_selftest_bounds",
            "ulysses_status_string", "ulysses_version")


class UlyssesError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {_STATUS.get(status, status)}")


_lib = None


def debug_build_selected() -> bool:
    """ULY_DEBUG_BUILD=1 in the environment selects the bounds-checked build
    of the library (compiled with -DULY_DEBUG) for this process."""
    return os.environ.get("ULY_DEBUG_BUILD", "") == "1"


def library_path() -> str:
    return _build_mod.DEBUG_SO_PATH if debug_build_selected() else _build_mod.SO_PATH


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load the shared library (it must have been built by ``build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"CUDA library not built: {path} is missing; run "
                               "`python -m long_context_sequence_head_gb300.build`")
        _build_mod.build(debug=debug_build_selected())
    lib = ctypes.CDLL(path)
    i64, i32, u64, vp, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_float
    sz = ctypes.c_size_t
    lib.ulysses_seq_to_head.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, vp]
    lib.ulysses_head_to_seq.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, vp]
    lib.ulysses_swap_batch.argtypes = [vp, i32, i64, i64, i32, i32, i32, vp]
    lib.ulysses_attn_workspace_size.argtypes = [i64, i64, i32, i32, i32, i32, i32, i32, i32]
    lib.ulysses_attn_workspace_size.restype = sz
    lib.ulysses_attn_tile_order.argtypes = [i64, i32, vp, i32, i32, vp]
    lib.ulysses_attn_fwd.argtypes = [vp] * 5 + [i64, i64, i32, i32, i32, i32, i32, vp, i32, f32, i32, vp, sz, vp]
    lib.ulysses_attn_bwd.argtypes = [vp] * 9 + [i64, i64, i32, i32, i32, i32, i32, vp, i32, f32, i32, vp, sz, vp]
    lib.ulysses_attn_fwd_seq.argtypes = lib.ulysses_attn_fwd.argtypes
    lib.ulysses_attn_bwd_seq.argtypes = lib.ulysses_attn_bwd.argtypes
    lib.ulysses_attn_bwd_noalloc.argtypes = [vp] * 9 + [i64, i64, i32, i32, i32, i32, i32, vp, i32, f32, i32, vp]
    lib.ulysses_ring_attn_workspace_size.argtypes = [i64, i64, i32, i32, i32, i32, i32, i32]
    lib.ulysses_ring_attn_workspace_size.restype = sz
    lib.ulysses_ring_attn_fwd.argtypes = [vp] * 5 + [i64, i64, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
    lib.ulysses_ring_attn_fwd.restype = i32
    lib.ulysses_ring_attn_bwd.argtypes = [vp] * 9 + [i64, i64, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
    lib.ulysses_ring_attn_bwd.restype = i32
    lib.ulysses_sharded_ce_workspace_size.argtypes = [i64, i64, i32]
    lib.ulysses_sharded_ce_workspace_size.restype = sz
    lib.ulysses_sharded_ce_loss.argtypes = [vp] * 6 + [i64, i64, i32, i32, i32, vp, sz, vp]
    lib.ulysses_sharded_ce_loss.restype = i32
    lib.ulysses_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.ulysses_set_wait_limit_ns.argtypes = [u64]
    lib.ulysses_selftest_wait_timeout.argtypes = [u64, vp]
    lib.ulysses_selftest_bounds.argtypes = [vp]
    lib.ulysses_status_string.argtypes = [i32]
    lib.ulysses_status_string.restype = ctypes.c_char_p
    lib.ulysses_version.restype = i32
    for name in ("ulysses_seq_to_head", "ulysses_head_to_seq", "ulysses_swap_batch", "ulysses_attn_fwd",
                 "ulysses_attn_bwd",
                 "ulysses_attn_bwd_noalloc", "ulysses_attn_fwd_seq", "ulysses_attn_bwd_seq",
                 "ulysses_get_device_status", "ulysses_set_wait_limit_ns", "ulysses_selftest_wait_timeout",
                 "ulysses_selftest_bounds", "ulysses_attn_tile_order"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def _check(fn: str, st: int):
    if st != ULY_OK:
        raise UlyssesError(fn, st)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ULY_BF16
    if t.dtype == torch.float32:
        return ULY_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev(*ts: torch.Tensor):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _attn_args(q, k, v, like_q=(), like_k=(), lse=None, lse_shape=None, shards=None):
    """The attention calls take every size from q and k; before any pointer
    reaches the library, the other tensors must have the shapes and dtypes
    include/ulysses.h states for them (a mismatch would be read or written
    out of bounds)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dim() != 5:
            raise ValueError(f"{name} must be 5-D [shards][B][tokens][heads][d], got {tuple(t.shape)}")
    if tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"v {tuple(v.shape)} must have the shape of k {tuple(k.shape)}")
    if k.shape[:3] != q.shape[:3] or k.shape[4] != q.shape[4]:
        raise ValueError(f"k {tuple(k.shape)} must match q {tuple(q.shape)} except in its head count")
    if shards is not None and q.shape[0] != shards:
        raise ValueError(f"the leading dimension of q must be P={shards}, got {q.shape[0]}")
    for t in (k, v) + tuple(like_q) + tuple(like_k):
        if t.dtype != q.dtype:
            raise ValueError(f"all attention tensors must share q's dtype {q.dtype}, got {t.dtype}")
    for t in like_q:
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"expected a tensor of q's shape {tuple(q.shape)}, got {tuple(t.shape)}")
    for t in like_k:
        if tuple(t.shape) != tuple(k.shape):
            raise ValueError(f"expected a tensor of k's shape {tuple(k.shape)}, got {tuple(t.shape)}")
    if lse is not None:
        if lse.dtype != torch.float32:
            raise ValueError(f"lse must be float32, got {lse.dtype}")
        if tuple(lse.shape) != tuple(lse_shape):
            raise ValueError(f"lse must have shape {tuple(lse_shape)}, got {tuple(lse.shape)}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _cu(cu_seqlens):
    if cu_seqlens is None:
        return None, 0, None
    arr = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    return arr.ctypes.data_as(ctypes.c_void_p), len(arr) - 1, arr


# ------------------------------------------------------------------ swaps

def ulysses_seq_to_head(x_seq: torch.Tensor, x_head: torch.Tensor, P: int, stream=None) -> torch.Tensor:
    """[P][B][N/P][H][d] -> [P][B][N][H/P][d] (see include/ulysses.h)."""
    _dev(x_seq, x_head)
    Ps, B, Np, H, d = x_seq.shape
    if Ps != P or tuple(x_head.shape) != (P, B, Np * P, H // P, d) or x_head.dtype != x_seq.dtype:
        raise ValueError("x_head must be [P][B][N][H/P][d] with the dtype of x_seq")
    _check("ulysses_seq_to_head", load().ulysses_seq_to_head(
        x_seq.data_ptr(), x_head.data_ptr(), B, Np * P, H, d, P, _dt(x_seq), _stream(stream)))
    return x_head


def ulysses_head_to_seq(x_head: torch.Tensor, x_seq: torch.Tensor, P: int, stream=None) -> torch.Tensor:
    """[P][B][N][H/P][d] -> [P][B][N/P][H][d] (see include/ulysses.h)."""
    _dev(x_head, x_seq)
    Ps, B, N, Hp, d = x_head.shape
    if Ps != P or tuple(x_seq.shape) != (P, B, N // P, Hp * P, d) or x_seq.dtype != x_head.dtype:
        raise ValueError("x_seq must be [P][B][N/P][H][d] with the dtype of x_head")
    _check("ulysses_head_to_seq", load().ulysses_head_to_seq(
        x_head.data_ptr(), x_seq.data_ptr(), B, N, Hp * P, d, P, _dt(x_head), _stream(stream)))
    return x_seq


class _SwapDesc(ctypes.Structure):
    _fields_ = [("src", ctypes.c_void_p), ("dst", ctypes.c_void_p), ("H", ctypes.c_int32),
                ("to_head", ctypes.c_int32)]


def ulysses_swap_batch(items, P: int, stream=None):
    """Up to four swaps in one launch (see include/ulysses.h).  items: a
    sequence of (src, dst, to_head); to_head=True takes a seq-layout src
    [P][B][N/P][H][d] to a head-layout dst [P][B][N][H/P][d], False the
    reverse.  All tensors share B, N, d, P and dtype."""
    items = list(items)
    if not 1 <= len(items) <= 4:
        raise ValueError("a swap batch holds 1 to 4 tensors")
    descs = (_SwapDesc * len(items))()
    shape = None
    dtype = None
    for i, (src, dst, to_head) in enumerate(items):
        _dev(src, dst)
        if to_head:
            Ps, B, Np, H, d = src.shape
            want = (P, B, Np * P, H // P, d)
            got = tuple(dst.shape)
        else:
            Ps, B, N_, Hp, d = src.shape
            Np, H = N_ // P, Hp * P
            want = (P, B, Np, H, d)
            got = tuple(dst.shape)
        if Ps != P or got != want or dst.dtype != src.dtype:
            raise ValueError(f"item {i}: expected a destination of shape {want} and the source dtype, got {got}")
        if shape is None:
            shape, dtype = (B, Np * P, d), src.dtype
        elif (B, Np * P, d) != shape or src.dtype != dtype:
            raise ValueError("all tensors of a batch share B, N, d and dtype")
        descs[i] = _SwapDesc(src.data_ptr(), dst.data_ptr(), H, 1 if to_head else 0)
    B, N, d = shape
    _check("ulysses_swap_batch", load().ulysses_swap_batch(
        ctypes.cast(descs, ctypes.c_void_p), len(items), B, N, d, P, ULY_BF16 if dtype == torch.bfloat16
        else ULY_FP32, _stream(stream)))


# ------------------------------------------------ all-to-all across GPUs

def _a2a_shapes(x, what):
    if x.dim() != 4 or x.shape[0] != 1:
        raise ValueError(f"{what} must be [1][tokens][heads][d] (batch 1), got {tuple(x.shape)}")
    if not x.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return x.shape[1], x.shape[2], x.shape[3]


def _a2a_out(out, shape, like, what):
    """A caller-supplied output buffer, checked, or a new one."""
    if out is None:
        return torch.empty(*shape, dtype=like.dtype, device=like.device)
    if (tuple(out.shape) != tuple(shape) or out.dtype != like.dtype or out.device != like.device
            or not out.is_contiguous()):
        raise ValueError(f"{what} must be a contiguous {tuple(shape)} tensor of {like.dtype} on {like.device}")
    return out


def ulysses_a2a_pack(x_local: torch.Tensor, P: int, out: Optional[torch.Tensor] = None, stream=None):
    """Send buffer of the seq->head all-to-all on one rank: this rank's
    sequence shard x_local [1][T][H][d] (its T tokens, all H heads) as P
    contiguous blocks [P][1][T][H/P][d], block s holding head block s for
    rank s.  It is the library's seq->head kernel applied to the rank's own
    shard seen as P sub-shards of T/P tokens (so T % P == 0)."""
    T, H, d = _a2a_shapes(x_local, "x_local")
    if T % P or H % P:
        raise ValueError(f"the local tokens ({T}) and the heads ({H}) must be multiples of P={P}")
    out = _a2a_out(out, (P, 1, T, H // P, d), x_local, "out")
    ulysses_seq_to_head(x_local.view(P, 1, T // P, H, d), out, P, stream)
    return out


def ulysses_a2a_unpack(recv: torch.Tensor, P: int, out: Optional[torch.Tensor] = None, stream=None):
    """Receive side of the head->seq all-to-all on one rank: recv [P][1][T][H/P][d]
    (block s = head block s of this rank's T tokens, from rank s) back to the
    sequence shard [1][T][H][d]: the library's head->seq kernel on the rank's
    own tokens."""
    if recv.dim() != 5 or not recv.is_contiguous():
        raise ValueError(f"recv must be a contiguous [P={P}][1][T][H/P][d] tensor, got {tuple(recv.shape)}")
    Ps, B, T, Hp, d = recv.shape
    if Ps != P or B != 1 or T % P:
        raise ValueError(f"recv must be [P={P}][1][T][H/P][d] with T % P == 0, got {tuple(recv.shape)}")
    out = _a2a_out(out, (1, T, Hp * P, d), recv, "out")
    ulysses_head_to_seq(recv, out.view(P, 1, T // P, Hp * P, d), P, stream)
    return out


def ulysses_all_to_all_seq_to_head(x_local: torch.Tensor, group=None, out: Optional[torch.Tensor] = None):
    """The first all-to-all of Ulysses across the P ranks of a process group
    (one GPU per rank; Transformers docs "Ulysses sequence parallelism", the
    all-to-all diagram; blog summary step 3): rank r holds tokens
    [r*T, (r+1)*T) of all H heads, x_local [1][T][H][d]; afterwards it holds
    all N = P*T tokens of heads [r*H/P, (r+1)*H/P), returned as the head
    shard [1][N][H/P][d] that the attention calls take (num_shards = 1).

    The local pack runs in the library's kernel; torch.distributed's
    all_to_all_single moves block s to rank s, each received block landing in
    this rank's own buffer.  Blocks arrive in source-rank order, which is
    token order, so the receive buffer is the head shard with no further
    copy.  Per rank (P-1)/P of the shard crosses the network: O(N d / P)."""
    import torch.distributed as dist
    P = dist.get_world_size(group)
    T, H, d = _a2a_shapes(x_local, "x_local")
    send = ulysses_a2a_pack(x_local, P)
    out = _a2a_out(out, (1, P * T, H // P, d), x_local, "out")
    dist.all_to_all_single(out.view(P, T * (H // P) * d), send.view(P, T * (H // P) * d), group=group)
    return out


def ulysses_all_to_all_head_to_seq(x_head: torch.Tensor, group=None, out: Optional[torch.Tensor] = None):
    """The second all-to-all (blog summary step 5), the inverse of
    ulysses_all_to_all_seq_to_head and its backward: this rank's head shard
    x_head [1][N][H/P][d] in, its sequence shard [1][N/P][H][d] out.  Block s
    of the head shard (the tokens of rank s) goes to rank s; the P received
    blocks (head block s of this rank's tokens, from rank s) are put back in
    the sequence layout by the library's head->seq kernel."""
    import torch.distributed as dist
    P = dist.get_world_size(group)
    N, Hp, d = _a2a_shapes(x_head, "x_head")
    if N % P:
        raise ValueError(f"the tokens ({N}) must be a multiple of P={P}")
    T = N // P
    recv = torch.empty(P, 1, T, Hp, d, dtype=x_head.dtype, device=x_head.device)
    dist.all_to_all_single(recv.view(P, T * Hp * d), x_head.view(P, T * Hp * d), group=group)
    return ulysses_a2a_unpack(recv, P, out)


# -------------------------------------------------------------- attention

def ulysses_attn_tile_order(N: int, causal: bool = True, cu_seqlens=None, for_bwd: bool = False) -> np.ndarray:
    """The order in which the bf16 kernels walk the 128-row tiles (see
    include/ulysses.h): every tile index once, longest walk first."""
    n = (int(N) + 127) // 128
    out = np.empty(max(n, 1), dtype=np.int32)
    cu_p, nd, _keep = _cu(cu_seqlens)
    _check("ulysses_attn_tile_order",
           load().ulysses_attn_tile_order(int(N), int(bool(causal)), cu_p, nd, int(bool(for_bwd)),
                                          out.ctypes.data_as(ctypes.c_void_p)))
    return out[:n]


def ulysses_attn_workspace_size(B: int, N: int, Hq_local: int, Hkv_local: int, d: int, num_shards: int,
                                num_docs: int, for_bwd: bool, dtype: torch.dtype) -> int:
    dt = ULY_BF16 if dtype == torch.bfloat16 else ULY_FP32
    return int(load().ulysses_attn_workspace_size(B, N, Hq_local, Hkv_local, d, num_shards, num_docs,
                                                  int(bool(for_bwd)), dt))


def _workspace(workspace, nbytes: int, device) -> torch.Tensor:
    if workspace is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace too small: need {nbytes} bytes")
    return workspace


def ulysses_attn_fwd(q, k, v, o, lse, causal: bool = True, cu_seqlens: Optional[Sequence[int]] = None,
                     softmax_scale: float = 0.0, workspace: Optional[torch.Tensor] = None, stream=None):
    """Attention forward over head shards; writes o and lse (see include/ulysses.h)."""
    _attn_args(q, k, v, like_q=(o,), lse=lse, lse_shape=(q.shape[0], q.shape[1], q.shape[3], q.shape[2]))
    _dev(q, k, v, o, lse)
    S, B, N, Hq, d = q.shape
    Hkv = k.shape[3]
    cu_p, nd, _keep = _cu(cu_seqlens)
    need = ulysses_attn_workspace_size(B, N, Hq, Hkv, d, S, nd, False, q.dtype)
    ws = _workspace(workspace, need, q.device)
    _check("ulysses_attn_fwd", load().ulysses_attn_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, N, Hq, Hkv, d, S,
        int(bool(causal)), cu_p, nd, float(softmax_scale), _dt(q), ws.data_ptr(),
        ws.numel() * ws.element_size(), _stream(stream)))
    return o, lse


def ulysses_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, causal: bool = True,
                     cu_seqlens: Optional[Sequence[int]] = None, softmax_scale: float = 0.0,
                     workspace: Optional[torch.Tensor] = None, stream=None):
    """Attention backward; writes dq, dk, dv (see include/ulysses.h)."""
    _attn_args(q, k, v, like_q=(o, dout, dq), like_k=(dk, dv), lse=lse,
               lse_shape=(q.shape[0], q.shape[1], q.shape[3], q.shape[2]))
    _dev(q, k, v, o, lse, dout, dq, dk, dv)
    S, B, N, Hq, d = q.shape
    Hkv = k.shape[3]
    cu_p, nd, _keep = _cu(cu_seqlens)
    need = ulysses_attn_workspace_size(B, N, Hq, Hkv, d, S, nd, True, q.dtype)
    ws = _workspace(workspace, need, q.device)
    _check("ulysses_attn_bwd", load().ulysses_attn_bwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, N, Hq, Hkv, d, S, int(bool(causal)), cu_p, nd,
        float(softmax_scale), _dt(q), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)))
    return dq, dk, dv


def ulysses_attn_fwd_seq(q_seq, k_seq, v_seq, o_seq, lse, P: int, causal: bool = True,
                         cu_seqlens: Optional[Sequence[int]] = None, softmax_scale: float = 0.0,
                         workspace: Optional[torch.Tensor] = None, stream=None):
    """Attention over all P head shards read from and written to the
    sequence-sharded layout [P][B][N/P][H][d] (no swaps); lse [P][B][Hq/P][N]."""
    _attn_args(q_seq, k_seq, v_seq, like_q=(o_seq,), lse=lse, shards=P,
               lse_shape=(P, q_seq.shape[1], q_seq.shape[3] // max(P, 1), q_seq.shape[2] * P))
    _dev(q_seq, k_seq, v_seq, o_seq, lse)
    Ps, B, Np, Hq, d = q_seq.shape
    Hkv = k_seq.shape[3]
    N = Np * P
    cu_p, nd, _keep = _cu(cu_seqlens)
    need = ulysses_attn_workspace_size(B, N, Hq // P, Hkv // P, d, P, nd, False, q_seq.dtype)
    ws = _workspace(workspace, need, q_seq.device)
    _check("ulysses_attn_fwd_seq", load().ulysses_attn_fwd_seq(
        q_seq.data_ptr(), k_seq.data_ptr(), v_seq.data_ptr(), o_seq.data_ptr(), lse.data_ptr(), B, N, Hq, Hkv,
        d, P, int(bool(causal)), cu_p, nd, float(softmax_scale), _dt(q_seq), ws.data_ptr(),
        ws.numel() * ws.element_size(), _stream(stream)))
    return o_seq, lse


def ulysses_attn_bwd_seq(q_seq, k_seq, v_seq, o_seq, lse, dout_seq, dq_seq, dk_seq, dv_seq, P: int,
                         causal: bool = True, cu_seqlens: Optional[Sequence[int]] = None,
                         softmax_scale: float = 0.0, workspace: Optional[torch.Tensor] = None, stream=None):
    """Backward of ulysses_attn_fwd_seq, all tensors in the sequence-sharded layout."""
    _attn_args(q_seq, k_seq, v_seq, like_q=(o_seq, dout_seq, dq_seq), like_k=(dk_seq, dv_seq), lse=lse,
               shards=P, lse_shape=(P, q_seq.shape[1], q_seq.shape[3] // max(P, 1), q_seq.shape[2] * P))
    _dev(q_seq, k_seq, v_seq, o_seq, lse, dout_seq, dq_seq, dk_seq, dv_seq)
    Ps, B, Np, Hq, d = q_seq.shape
    Hkv = k_seq.shape[3]
    N = Np * P
    cu_p, nd, _keep = _cu(cu_seqlens)
    need = ulysses_attn_workspace_size(B, N, Hq // P, Hkv // P, d, P, nd, True, q_seq.dtype)
    ws = _workspace(workspace, need, q_seq.device)
    _check("ulysses_attn_bwd_seq", load().ulysses_attn_bwd_seq(
        q_seq.data_ptr(), k_seq.data_ptr(), v_seq.data_ptr(), o_seq.data_ptr(), lse.data_ptr(),
        dout_seq.data_ptr(), dq_seq.data_ptr(), dk_seq.data_ptr(), dv_seq.data_ptr(), B, N, Hq, Hkv, d, P,
        int(bool(causal)), cu_p, nd, float(softmax_scale), _dt(q_seq), ws.data_ptr(),
        ws.numel() * ws.element_size(), _stream(stream)))
    return dq_seq, dk_seq, dv_seq


def ulysses_attn_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, causal: bool = True,
                             cu_seqlens: Optional[Sequence[int]] = None, softmax_scale: float = 0.0,
                             stream=None):
    """Attention backward without a workspace, for callers that cannot
    allocate device memory; its scratch is a fixed 64 MiB array inside the
    library (see include/ulysses.h for the limits and the ordering rule).
    The call runs with q's device current, since the library takes the
    scratch address of the current device."""
    _attn_args(q, k, v, like_q=(o, dout, dq), like_k=(dk, dv), lse=lse,
               lse_shape=(q.shape[0], q.shape[1], q.shape[3], q.shape[2]))
    _dev(q, k, v, o, lse, dout, dq, dk, dv)
    for t in (k, v, o, lse, dout, dq, dk, dv):
        if t.device != q.device:
            raise ValueError("all tensors must live on q's device")
    if isinstance(stream, torch.cuda.Stream) and stream.device != q.device:
        raise ValueError("the stream must belong to q's device")
    S, B, N, Hq, d = q.shape
    Hkv = k.shape[3]
    cu_p, nd, _keep = _cu(cu_seqlens)
    with torch.cuda.device(q.device):
        _check("ulysses_attn_bwd_noalloc", load().ulysses_attn_bwd_noalloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, N, Hq, Hkv, d, S, int(bool(causal)), cu_p, nd,
            float(softmax_scale), _dt(q), _stream(stream)))
    return dq, dk, dv


# -------------------------------------------------------- ring attention

def ulysses_ring_attn_fwd(q_seq, k_seq, v_seq, o_seq, lse, P: int, causal: bool = True,
                          softmax_scale: float = 0.0, workspace: Optional[torch.Tensor] = None, stream=None):
    """Ring attention over P chunks of the sequence-sharded layout; lse [P][B][Hq][N/P]."""
    _attn_args(q_seq, k_seq, v_seq, like_q=(o_seq,), lse=lse, shards=P,
               lse_shape=(P, q_seq.shape[1], q_seq.shape[3], q_seq.shape[2]))
    _dev(q_seq, k_seq, v_seq, o_seq, lse)
    Ps, B, Np, Hq, d = q_seq.shape
    Hkv = k_seq.shape[3]
    N = Np * P
    need = int(load().ulysses_ring_attn_workspace_size(B, N, Hq, Hkv, d, P, 0, _dt(q_seq)))
    ws = _workspace(workspace, need, q_seq.device)
    _check("ulysses_ring_attn_fwd", load().ulysses_ring_attn_fwd(
        q_seq.data_ptr(), k_seq.data_ptr(), v_seq.data_ptr(), o_seq.data_ptr(), lse.data_ptr(), B, N, Hq, Hkv,
        d, P, int(bool(causal)), float(softmax_scale), _dt(q_seq), ws.data_ptr(),
        ws.numel() * ws.element_size(), _stream(stream)))
    return o_seq, lse


def ulysses_ring_attn_bwd(q_seq, k_seq, v_seq, o_seq, lse, dout_seq, dq_seq, dk_seq, dv_seq, P: int,
                          causal: bool = True, softmax_scale: float = 0.0,
                          workspace: Optional[torch.Tensor] = None, stream=None):
    """Backward of ulysses_ring_attn_fwd (final o and lse)."""
    _attn_args(q_seq, k_seq, v_seq, like_q=(o_seq, dout_seq, dq_seq), like_k=(dk_seq, dv_seq), lse=lse,
               shards=P, lse_shape=(P, q_seq.shape[1], q_seq.shape[3], q_seq.shape[2]))
    _dev(q_seq, k_seq, v_seq, o_seq, lse, dout_seq, dq_seq, dk_seq, dv_seq)
    Ps, B, Np, Hq, d = q_seq.shape
    Hkv = k_seq.shape[3]
    N = Np * P
    need = int(load().ulysses_ring_attn_workspace_size(B, N, Hq, Hkv, d, P, 1, _dt(q_seq)))
    ws = _workspace(workspace, need, q_seq.device)
    _check("ulysses_ring_attn_bwd", load().ulysses_ring_attn_bwd(
        q_seq.data_ptr(), k_seq.data_ptr(), v_seq.data_ptr(), o_seq.data_ptr(), lse.data_ptr(),
        dout_seq.data_ptr(), dq_seq.data_ptr(), dk_seq.data_ptr(), dv_seq.data_ptr(), B, N, Hq, Hkv, d, P,
        int(bool(causal)), float(softmax_scale), _dt(q_seq), ws.data_ptr(), ws.numel() * ws.element_size(),
        _stream(stream)))
    return dq_seq, dk_seq, dv_seq


# ---------------------------------------------------------- sharded loss

def ulysses_sharded_ce_loss(logits, labels, P: int, dlogits: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None, stream=None,
                            outputs: Optional[Sequence[torch.Tensor]] = None):
    """Shifted next-token CE per rank and its good-token-weighted aggregation.

    logits [P][B][N/P][V] (bf16/fp32), labels [P][B][N/P] int64 (unshifted,
    -100 = ignored).  Returns (shard_loss [P] fp32, shard_good [P] int64,
    total [1] fp32) on the device; fills dlogits (like logits) if given.
    `outputs` may supply those three tensors (else they are allocated).
    """
    if logits.dim() != 4 or logits.shape[0] != P:
        raise ValueError(f"logits must be [P={P}][B][N/P][V], got {tuple(logits.shape)}")
    if dlogits is not None and (tuple(dlogits.shape) != tuple(logits.shape) or dlogits.dtype != logits.dtype):
        raise ValueError("dlogits must have the shape and dtype of logits")
    _dev(logits, labels)
    if dlogits is not None:
        _dev(dlogits)
    Ps, B, Np, V = logits.shape
    N = Np * P
    if labels.dtype != torch.int64 or tuple(labels.shape) != (P, B, Np):
        raise ValueError("labels must be int64 [P][B][N/P]")
    dev = logits.device
    if outputs is None:
        shard_loss = torch.empty(P, dtype=torch.float32, device=dev)
        shard_good = torch.empty(P, dtype=torch.int64, device=dev)
        total = torch.empty(4, dtype=torch.float32, device=dev)
    else:
        shard_loss, shard_good, total = outputs
        if (shard_loss.dtype != torch.float32 or shard_loss.numel() != P or shard_good.dtype != torch.int64
                or shard_good.numel() != P or total.dtype != torch.float32 or total.numel() < 1):
            raise ValueError("outputs must be (fp32 [P], int64 [P], fp32 [>=1])")
        _dev(shard_loss, shard_good, total)
    need = int(load().ulysses_sharded_ce_workspace_size(B, N, P))
    ws = _workspace(workspace, need, dev)
    _check("ulysses_sharded_ce_loss", load().ulysses_sharded_ce_loss(
        logits.data_ptr(), labels.data_ptr(), dlogits.data_ptr() if dlogits is not None else None,
        shard_loss.data_ptr(), shard_good.data_ptr(), total.data_ptr(), B, N, V, P, _dt(logits),
        ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)))
    return shard_loss, shard_good, total[:1]


# ------------------------------------------------------------ diagnostics

def ulysses_get_device_status(stream=None):
    """Synchronise the stream, read and clear the device status.  Returns (status, site)."""
    site = ctypes.c_uint32(0)
    st = load().ulysses_get_device_status(_stream(stream), ctypes.byref(site))
    return int(st), int(site.value)


def ulysses_set_wait_limit_ns(limit_ns: int) -> None:
    _check("ulysses_set_wait_limit_ns", load().ulysses_set_wait_limit_ns(int(limit_ns)))


def ulysses_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check("ulysses_selftest_wait_timeout", load().ulysses_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def ulysses_selftest_bounds(stream=None) -> int:
    """Debug build: make one bounds check fail without touching memory
    (returns the call's status; the release build answers ULY_ERR_UNSUPPORTED)."""
    return int(load().ulysses_selftest_bounds(_stream(stream)))


def ulysses_status_string(status: int) -> str:
    return load().ulysses_status_string(int(status)).decode()


def ulysses_version() -> int:
    return int(load().ulysses_version())
