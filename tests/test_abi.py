"""C-ABI checks that need no GPU: the library loads, exports every symbol
``include/ulysses.h`` declares, and rejects invalid arguments on the host
before launching anything (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

INVALID, UNSUPPORTED, MISALIGNED, OVERLAP, WORKSPACE = 1, 2, 3, 4, 7
BF16, FP32 = 0, 1


def _declared():
    src = open(os.path.join(ROOT, "include", "ulysses.h")).read()
    return sorted(set(re.findall(r"\b(ulysses_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(uly):
    lib = uly.load()
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(uly.EXPORTED) == names


def test_version_and_strings(uly):
    assert uly.ulysses_version() == 100
    for code in range(10):
        assert uly.ulysses_status_string(code)
    assert uly.ulysses_status_string(0) == "ok"


def test_release_build_has_no_bounds_selftest(uly):
    """The bounds checks exist only in the debug build; the release library
    answers its self-test with ULY_ERR_UNSUPPORTED and launches nothing."""
    if uly.debug_build_selected():
        pytest.skip("this process runs the debug build")
    assert uly.load().ulysses_selftest_bounds(None) == UNSUPPORTED


def test_debug_build_exports_every_declared_symbol(uly):
    from long_context_sequence_head_gb300 import build as b
    lib = ctypes.CDLL(b.build(debug=True))
    for n in _declared():
        assert hasattr(lib, n), n


def _swap(lib, a, b, B, N, H, d, P, dt=BF16):
    return lib.ulysses_seq_to_head(a, b, B, N, H, d, P, dt, None)


def test_swap_validation(uly):
    lib = uly.load()
    a, b = 1 << 20, 1 << 40  # never dereferenced: every call below fails validation
    assert _swap(lib, None, b, 1, 8, 4, 64, 2) == INVALID
    assert _swap(lib, a, b, 0, 8, 4, 64, 2) == INVALID          # empty batch
    assert _swap(lib, a, b, 1, 0, 4, 64, 2) == INVALID          # empty sequence
    assert _swap(lib, a, b, 1, 9, 4, 64, 2) == INVALID          # N not padded to a multiple of P
    assert _swap(lib, a, b, 1, 8, 6, 64, 4) == INVALID          # heads not divisible by P
    assert _swap(lib, a, b, 1, 8, 2, 64, 4) == INVALID          # P > H
    assert _swap(lib, a, b, 1, 8, 4, 96, 2) == UNSUPPORTED      # head_dim
    assert _swap(lib, a + 8, b, 1, 8, 4, 64, 2) == MISALIGNED
    assert _swap(lib, a, a + 64, 1, 8, 4, 64, 2) == OVERLAP
    assert _swap(lib, a, b, 1, 8, 4, 64, 2, dt=7) == INVALID


def _batch(lib, uly, entries, B, N, d, P, dt=BF16):
    descs = (uly._SwapDesc * max(len(entries), 1))()
    for i, (src, dst, H, to_head) in enumerate(entries):
        descs[i] = uly._SwapDesc(src, dst, H, to_head)
    return lib.ulysses_swap_batch(ctypes.cast(descs, ctypes.c_void_p), len(entries), B, N, d, P, dt, None)


def test_swap_batch_validation(uly):
    lib = uly.load()
    a, b, c, e = 1 << 20, 1 << 40, 1 << 41, 1 << 42  # never dereferenced
    assert lib.ulysses_swap_batch(None, 1, 1, 8, 64, 2, BF16, None) == INVALID
    assert _batch(lib, uly, [], 1, 8, 64, 2) == INVALID                                  # empty batch
    assert _batch(lib, uly, [(a, b, 4, 1)] * 5, 1, 8, 64, 2) == INVALID                  # more than four
    assert _batch(lib, uly, [(a, b, 4, 1), (c, e, 6, 1)], 1, 8, 64, 4) == INVALID        # 6 heads, P = 4
    assert _batch(lib, uly, [(a, b, 4, 2)], 1, 8, 64, 2) == INVALID                      # direction flag
    assert _batch(lib, uly, [(a, b, 4, 1), (c + 8, e, 4, 0)], 1, 8, 64, 2) == MISALIGNED
    assert _batch(lib, uly, [(a, b, 4, 1), (c, b, 4, 1)], 1, 8, 64, 2) == OVERLAP        # two writers
    assert _batch(lib, uly, [(a, b, 4, 1), (b, c, 4, 0)], 1, 8, 64, 2) == OVERLAP        # one reads the other's output
    assert _batch(lib, uly, [(a, b, 4, 1), (c, e, 4, 1)], 1, 8, 96, 2) == UNSUPPORTED    # head_dim


def test_head_divisibility_golden(uly):
    """32 heads support SP sizes 1, 2, 4, 8, 16, 32 (fixture cites the page)."""
    lib = uly.load()
    spec = {}
    for line in open(os.path.join(GOLDEN, "head_divisibility_h32.txt")):
        if line.strip() and not line.startswith("#"):
            k, *vals = line.split()
            spec[k] = [int(v) for v in vals]
    H = spec["H"][0]
    a, b = 1 << 20, 1 << 40
    for P in spec["invalid"]:
        assert lib.ulysses_seq_to_head(a, b, 1, 64 * 64, H, 128, P, BF16, None) in (INVALID,), P
    # valid P pass validation: with a misaligned pointer the call must stop at
    # the alignment check, proving the divisibility checks accepted P
    for P in spec["valid"]:
        assert lib.ulysses_seq_to_head(a + 8, b, 1, 64 * 64, H, 128, P, BF16, None) == MISALIGNED, P


def test_attn_validation(uly):
    lib = uly.load()
    p = 1 << 20
    ws = uly.ulysses_attn_workspace_size
    import torch
    need = ws(1, 256, 8, 2, 128, 4, 0, False, torch.bfloat16)
    assert need > 0
    assert ws(1, 256, 8, 3, 128, 4, 0, False, torch.bfloat16) == 0  # Hq % Hkv != 0
    assert ws(1, 256, 8, 2, 64, 4, 0, False, torch.bfloat16) == 0   # bf16 needs d = 128
    assert ws(1, 256, 8, 2, 64, 4, 0, True, torch.float32) > 0
    bwd = ws(1, 1000, 8, 2, 128, 1, 3, True, torch.bfloat16)
    assert bwd >= 1024 * 8 * 4 * (2 + 128)  # lse2 + D + dq accumulator over padded rows

    def fwd(B=1, N=256, Hq=8, Hkv=2, d=128, S=1, causal=1, cu=None, nd=0, dt=BF16, wsb=1 << 30, q=p):
        cu_p = None
        if cu is not None:
            arr = (ctypes.c_int32 * len(cu))(*cu)
            cu_p = ctypes.cast(arr, ctypes.c_void_p)
        return lib.ulysses_attn_fwd(q, p, p, p, p, B, N, Hq, Hkv, d, S, causal, cu_p, nd, 0.0, dt, p, wsb, None)

    assert fwd(Hkv=3) == INVALID
    assert fwd(N=0) == INVALID
    assert fwd(causal=2) == INVALID
    assert fwd(d=64) == UNSUPPORTED
    assert fwd(d=80, dt=FP32) == UNSUPPORTED
    assert fwd(cu=[0, 100, 256], nd=2, q=p + 4) == MISALIGNED     # valid docs, stops at alignment
    assert fwd(cu=[0, 100, 255], nd=2) == INVALID                 # last offset != N
    assert fwd(cu=[1, 100, 256], nd=2) == INVALID                 # first offset != 0
    assert fwd(cu=[0, 200, 100, 256], nd=3) == INVALID            # decreasing
    assert fwd(nd=2) == INVALID                                   # docs count without offsets
    assert fwd(wsb=16) == WORKSPACE
    assert lib.ulysses_attn_fwd(None, p, p, p, p, 1, 256, 8, 2, 128, 1, 1, None, 0, 0.0, BF16, p,
                                1 << 30, None) == INVALID


def test_seq_layout_validation(uly):
    lib = uly.load()
    p = 1 << 20

    def fwd_seq(B=1, N=1024, Hq=8, Hkv=4, d=128, P=4, dt=BF16, q=p):
        return lib.ulysses_attn_fwd_seq(q, p, p, p, p, B, N, Hq, Hkv, d, P, 1, None, 0, 0.0, dt, p, 1 << 30, None)

    assert fwd_seq(N=1026) == INVALID            # N not a multiple of P
    assert fwd_seq(Hkv=2) == INVALID             # KV heads not divisible by P
    assert fwd_seq(Hq=6, Hkv=4, P=2) == INVALID  # local GQA group not integral
    assert fwd_seq(N=4 * 200) == UNSUPPORTED     # bf16 tile would straddle two shards
    assert fwd_seq(N=4 * 200, dt=FP32, d=64, q=p + 4) == MISALIGNED   # fp32 has no tile rule
    assert fwd_seq(q=p + 4) == MISALIGNED


def test_ring_validation(uly):
    lib = uly.load()
    p = 1 << 20
    assert lib.ulysses_ring_attn_workspace_size(1, 1024, 8, 2, 128, 4, 1, BF16) > 0
    assert lib.ulysses_ring_attn_workspace_size(1, 1026, 8, 2, 128, 4, 1, BF16) == 0
    call = lambda N=1024, Hq=8, Hkv=2, d=128, P=4, dt=BF16, q=p, wsb=1 << 34: lib.ulysses_ring_attn_fwd(
        q, p, p, p, p, 1, N, Hq, Hkv, d, P, 1, 0.0, dt, p, wsb, None)
    assert call(N=1026) == INVALID
    assert call(Hkv=3) == INVALID
    assert call(d=64) == UNSUPPORTED
    assert call(q=p + 8) == MISALIGNED
    assert call(wsb=64) == WORKSPACE


def test_sharded_ce_validation(uly):
    lib = uly.load()
    p = 1 << 20
    ws = lib.ulysses_sharded_ce_workspace_size
    assert ws(1, 64, 4) > 0 and ws(1, 65, 4) == 0
    call = lambda N=64, P=4, V=100, dt=BF16, lg=p, dl=None, wsb=1 << 30: lib.ulysses_sharded_ce_loss(
        lg, p, dl, p, p, p, 1, N, V, P, dt, p, wsb, None)
    assert call(N=65) == INVALID          # not padded to a multiple of P
    assert call(V=0) == INVALID
    assert call(lg=p + 2) == MISALIGNED
    assert call(dl=p) == OVERLAP           # gradient would overwrite the logits
    assert call(wsb=8) == WORKSPACE


def test_wait_limit_validation(uly):
    lib = uly.load()
    assert lib.ulysses_set_wait_limit_ns(10) == INVALID
    assert lib.ulysses_selftest_wait_timeout(10, None) == INVALID
    assert lib.ulysses_set_wait_limit_ns(2_000_000_000) == 0
