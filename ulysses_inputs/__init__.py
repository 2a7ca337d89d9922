"""Seeded synthetic inputs for the Ulysses swap + attention path.

This module is shared by the fp64 oracle (``oracle/``) and the CUDA path
(``long_context_sequence_head_gb300``).  It holds no arithmetic of the method:
it only draws random numbers, builds document-length lists and names the
workloads.  Neither side imports the other; both import this.

Workloads (all causal, softmax scale 1/sqrt(head_dim), Q/K/V/dO ~ N(0, 1)):

* ``tiny_fp32_n256``      B=1, N=256,  P=2, 4 Q heads / 4 KV heads, d=64, fp32.
* ``qwen3_4b_n8192``      B=1, N=8192, P=4, 32 Q / 8 KV heads (GQA group 4), d=128, bf16.
* ``qwen3_4b_n65536``     same heads, N=65536.
* ``packed_docs_n32768``  same heads, N=32768 made of documents with lengths
                          uniform on [512, 8192], the last one truncated to fill N.
* ``single_shard_n1m``    same heads, N=2**20, P=8: one head shard holds
                          4 Q heads and 1 KV head.

The Qwen3-4B head shapes and the 64K/SP=4 setting stand in for the pages'
Qwen3-4B on Gutenberg-English benchmark (Hugging Face Ulysses blog summary,
"Performance Benchmarks"); no dataset or weights are used.

Layouts follow the Ulysses statement of the problem ("Ulysses sequence
parallelism", the all-to-all diagram): the sequence-sharded buffer is P
contiguous shards ``[P][B][N/P][H][d]``; the head-sharded buffer is
``[P][B][N][H/P][d]``.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, List, Optional

import numpy as np
import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "doc_lengths",
    "cu_seqlens_from_lengths",
    "draw_seq_inputs",
    "draw_labels_logits",
    "sha256_of",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    N: int
    P: int
    Hq: int
    Hkv: int
    d: int
    dtype: str  # "bf16" or "fp32"
    causal: bool = True
    packed_docs: bool = False
    # number of head shards the attention step is timed/checked on
    # (None = all P shards)
    attn_shards: Optional[int] = None

    @property
    def Hp(self) -> int:
        return self.Hq // self.P

    @property
    def Hkvp(self) -> int:
        return self.Hkv // self.P

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def shards_timed(self) -> int:
        return self.P if self.attn_shards is None else self.attn_shards

    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_fp32_n256", 1, 256, 2, 4, 4, 64, "fp32"),
        Workload("qwen3_4b_n8192", 1, 8192, 4, 32, 8, 128, "bf16"),
        Workload("qwen3_4b_n65536", 1, 65536, 4, 32, 8, 128, "bf16"),
        Workload("packed_docs_n32768", 1, 32768, 4, 32, 8, 128, "bf16", packed_docs=True),
        Workload("single_shard_n1m", 1, 1 << 20, 8, 32, 8, 128, "bf16", attn_shards=1),
    ]
}


def doc_lengths(N: int, P: int, seed: int, lo: int = 512, hi: int = 8192) -> List[int]:
    """Document lengths for a packed batch of total length N.

    Lengths are integers uniform on [lo, hi] inclusive, drawn in order until
    their sum reaches N; the last one is cut so the sum is exactly N.  The
    total is then padded to a multiple of P with one trailing padding
    document (TRL's ``pad_to_multiple_of=sp_size`` in the pages' packing
    discussion).  With N % P == 0 no padding document appears.
    """
    rng = np.random.default_rng(seed)
    out: List[int] = []
    total = 0
    while total < N:
        L = int(rng.integers(lo, hi + 1))
        L = min(L, N - total)
        out.append(L)
        total += L
    pad = (-total) % P
    if pad:
        out.append(pad)
    return out


def cu_seqlens_from_lengths(lengths: List[int]) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu


def draw_seq_inputs(w: Workload, seed: int, device: str = "cpu",
                    want_dout: bool = True, P: Optional[int] = None,
                    N: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Draw Q, K, V (and dO) in the sequence-sharded layout.

    Values are N(0, 1) in fp32 from one seeded generator in the fixed order
    Q, K, V, dO, then rounded to the workload dtype (round-to-nearest-even for
    bf16).  Shapes: Q/dO ``[P][B][N/P][Hq][d]``, K/V ``[P][B][N/P][Hkv][d]``.
    ``device="cuda"`` draws on the GPU (used for the large workloads).
    """
    P = w.P if P is None else P
    N = w.N if N is None else N
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt = w.torch_dtype()
    shape_q = (P, w.B, N // P, w.Hq, w.d)
    shape_kv = (P, w.B, N // P, w.Hkv, w.d)
    out = {}
    for name, shape in (("q", shape_q), ("k", shape_kv), ("v", shape_kv)) + (
            (("dout", shape_q),) if want_dout else ()):
        t = torch.empty(shape, dtype=torch.float32, device=device)
        t.normal_(0.0, 1.0, generator=gen)
        out[name] = t.to(dt)
        del t
    return out


def draw_labels_logits(N: int, V: int, seed: int, ignore_frac: float = 0.3):
    """Random logits [N][V] (fp64) and labels [N] (int64, -100 = ignored)."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((N, V))
    labels = rng.integers(0, V, size=N).astype(np.int64)
    labels[rng.random(N) < ignore_frac] = -100
    return logits, labels


def sha256_of(*tensors: torch.Tensor) -> str:
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()
