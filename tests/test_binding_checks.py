"""The Python binding refuses mismatched attention arguments before any
pointer reaches the library (CPU only: the checks run before the device
check, so CPU tensors exercise them)."""
import pytest
import torch

import long_context_sequence_head_gb300 as uly


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


S, B, N, Hq, Hkv, d = 2, 1, 64, 4, 2, 128


def _fwd_args():
    return dict(q=_t(S, B, N, Hq, d), k=_t(S, B, N, Hkv, d), v=_t(S, B, N, Hkv, d), o=_t(S, B, N, Hq, d),
                lse=_t(S, B, Hq, N, dtype=torch.float32))


def test_consistent_arguments_reach_the_device_check():
    with pytest.raises(ValueError, match="CUDA device"):
        uly.ulysses_attn_fwd(**_fwd_args())


@pytest.mark.parametrize("name,bad,msg", [
    ("kv", _t(S, B, N + 1, Hkv, d), "except in its head count"),
    ("v", _t(S, B, N, Hkv + 2, d), "shape of k"),
    ("o", _t(S, B, N, Hq, 64), "q's shape"),
    ("o", _t(S, B, N, Hq, d, dtype=torch.float32), "dtype"),
    ("lse", _t(S, B, N, Hq, dtype=torch.float32), "lse must have shape"),
    ("lse", _t(S, B, Hq, N), "float32"),
    ("q", _t(S, B, N, Hq * d), "5-D"),
])
def test_forward_mismatch_is_refused(name, bad, msg):
    args = _fwd_args()
    for key in (("k", "v") if name == "kv" else (name,)):
        args[key] = bad
    with pytest.raises(ValueError, match=msg):
        uly.ulysses_attn_fwd(**args)


def test_backward_gradient_shapes_are_checked():
    a = _fwd_args()
    dq, dk, dv, do = _t(S, B, N, Hq, d), _t(S, B, N, Hkv, d), _t(S, B, N, Hkv, d), _t(S, B, N, Hq, d)
    with pytest.raises(ValueError, match="k's shape"):
        uly.ulysses_attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], do, dq, _t(S, B, N, Hq, d), dv)
    with pytest.raises(ValueError, match="q's shape"):
        uly.ulysses_attn_bwd_noalloc(a["q"], a["k"], a["v"], a["o"], a["lse"], _t(S, B, N // 2, Hq, d), dq, dk, dv)
    with pytest.raises(ValueError, match="CUDA device"):
        uly.ulysses_attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], do, dq, dk, dv)


def test_seq_and_ring_layouts():
    P, Np = 2, 32
    q, k, v, o = _t(P, B, Np, Hq, d), _t(P, B, Np, Hkv, d), _t(P, B, Np, Hkv, d), _t(P, B, Np, Hq, d)
    lse_seq = _t(P, B, Hq // P, Np * P, dtype=torch.float32)   # [P][B][Hq/P][N]
    lse_ring = _t(P, B, Hq, Np, dtype=torch.float32)           # [P][B][Hq][N/P]
    with pytest.raises(ValueError, match="CUDA device"):
        uly.ulysses_attn_fwd_seq(q, k, v, o, lse_seq, P)
    with pytest.raises(ValueError, match="lse must have shape"):
        uly.ulysses_attn_fwd_seq(q, k, v, o, lse_ring, P)
    with pytest.raises(ValueError, match="CUDA device"):
        uly.ulysses_ring_attn_fwd(q, k, v, o, lse_ring, P)
    with pytest.raises(ValueError, match="lse must have shape"):
        uly.ulysses_ring_attn_fwd(q, k, v, o, lse_seq, P)
    with pytest.raises(ValueError, match="leading dimension"):
        uly.ulysses_attn_fwd_seq(q, k, v, o, lse_seq, 4)


def test_sharded_loss_arguments():
    P, Np, V = 2, 8, 64
    logits = _t(P, B, Np, V)
    labels = torch.zeros(P, B, Np, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA device"):
        uly.ulysses_sharded_ce_loss(logits, labels, P, dlogits=_t(P, B, Np, V))
    with pytest.raises(ValueError, match="shape and dtype of logits"):
        uly.ulysses_sharded_ce_loss(logits, labels, P, dlogits=_t(P, B, Np, V - 8))
    with pytest.raises(ValueError, match="shape and dtype of logits"):
        uly.ulysses_sharded_ce_loss(logits, labels, P, dlogits=_t(P, B, Np, V, dtype=torch.float32))
    with pytest.raises(ValueError, match="logits must be"):
        uly.ulysses_sharded_ce_loss(logits, labels, 4)


def test_all_to_all_helpers_check_their_buffers():
    """The exchange's pack/unpack refuse non-contiguous inputs and outputs of
    the wrong shape, dtype or device before any kernel is reached."""
    import long_context_sequence_head_gb300 as uly
    x = torch.zeros(1, 8, 4, 64)
    with pytest.raises(ValueError):
        uly.ulysses_a2a_pack(x.transpose(1, 2), 2)                      # not contiguous
    with pytest.raises(ValueError):
        uly.ulysses_a2a_pack(torch.zeros(2, 8, 4, 64), 2)               # batch 2
    with pytest.raises(ValueError):
        uly.ulysses_a2a_pack(x, 2, out=torch.zeros(2, 1, 8, 2, 32))     # wrong out shape
    with pytest.raises(ValueError):
        uly.ulysses_a2a_pack(x, 2, out=torch.zeros(2, 1, 8, 2, 64, dtype=torch.float64))
    with pytest.raises(ValueError):
        uly.ulysses_a2a_unpack(torch.zeros(2, 1, 7, 2, 64), 2)          # T not a multiple of P
