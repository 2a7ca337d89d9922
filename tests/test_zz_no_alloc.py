"""The no-allocation backward (ulysses_attn_bwd_noalloc) against the regular
one (ulysses_attn_bwd with a caller-allocated workspace).

Callers such as allocator hooks, fixed-pool processes or plugins handed only
their tensors cannot allocate the backward's scratch; this entry point keeps
that scratch in a fixed device array inside the library.  The test calls it
through the C ABI twice in a row with different inputs -- the second call
sees the first call's leftovers in the shared array -- and checks both
results against the regular entry point within the parity tolerance of the
dtype (bf16 and fp32), and that the later call leaves the device's free
memory unchanged.  It also checks that sizes beyond the array are refused.
Kept in its own file so pytest collects it last.
"""
import ctypes

import pytest
import torch

from parity_utils import REL_TOL, rel_fro

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 8


def _inputs(seed, S, N, Hq, Hkv, d, dtype):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda H: torch.randn(S, 1, N, H, d, device="cuda", generator=g).to(dtype)
    return mk(Hq), mk(Hkv), mk(Hkv), mk(Hq)


def _call_noalloc(lib, q, k, v, o, lse, do, dq, dk, dv, cu=None):
    S, B, N, Hq, d = q.shape
    Hkv = k.shape[3]
    cu_p, nd = None, 0
    if cu is not None:
        arr = (ctypes.c_int32 * len(cu))(*cu)
        cu_p, nd = ctypes.cast(arr, ctypes.c_void_p), len(cu) - 1
    dt = 0 if q.dtype == torch.bfloat16 else 1
    return lib.ulysses_attn_bwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, N, Hq, Hkv, d, S, 1, cu_p, nd, 0.0, dt,
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("S,N,Hq,Hkv,d,dtype,cu", [
    (2, 1000, 4, 1, 128, torch.bfloat16, None),
    (1, 1300, 8, 2, 128, torch.bfloat16, [0, 5, 700, 1300]),
    (2, 256, 4, 4, 64, torch.float32, None),           # the fp32 path keeps only D in the array
])
def test_noalloc_matches_workspace_entry_point(uly, S, N, Hq, Hkv, d, dtype, cu):
    lib = uly.load()
    tag = "bf16" if dtype == torch.bfloat16 else "fp32"
    for call, seed in enumerate((10, 20)):
        q, k, v, do = _inputs(seed + S, S, N, Hq, Hkv, d, dtype)
        o = torch.empty_like(q)
        lse = torch.empty(S, 1, Hq, N, dtype=torch.float32, device="cuda")
        uly.ulysses_attn_fwd(q, k, v, o, lse, cu_seqlens=cu)
        ref = [torch.empty_like(x) for x in (q, k, v)]
        uly.ulysses_attn_bwd(q, k, v, o, lse, do, *ref, cu_seqlens=cu)
        got = [torch.full_like(x, float("nan")) for x in (q, k, v)]
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _call_noalloc(lib, q, k, v, o, lse, do, *got, cu=cu) == 0
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert uly.ulysses_get_device_status()[0] == 0
        if call > 0:
            # the module holding the array is loaded by the first call; later
            # calls take no device memory at all
            assert free_after == free_before, (free_before, free_after)
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(a.float()).all(), (call, name)
            assert rel_fro(a, b) <= REL_TOL[tag], (call, name, rel_fro(a, b))


def test_noalloc_rejects_sizes_beyond_its_scratch(uly):
    lib = uly.load()
    p = 1 << 20  # never dereferenced: the call must refuse before launching
    st = lib.ulysses_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 65536, 8, 2, 128, 4, 1, None, 0, 0.0, 0,
                                      None)
    assert st == SCRATCH_LIMIT
    assert uly.ulysses_status_string(st).startswith("sizes exceed")
