"""The Python binding's decode calls check every shape before any device
check or launch (CPU only). A short seqlens, out or cor would otherwise let
the kernels read or write past the end of a buffer."""
import pytest
import torch

from parametrized_local_linear_gb300 import (plx_decode_fwd, plx_decode_fwd_cor,
                                             plx_decode_fwd_noalloc)


def _decode_args(B=3, Hq=4, Hkv=2, d=128, T=50):
    bf = torch.bfloat16
    return (torch.zeros(B, Hq, d, dtype=bf), torch.zeros(B, Hq, d, dtype=bf),
            torch.zeros(T, Hkv, d, dtype=bf), torch.zeros(T, Hkv, d, dtype=bf),
            torch.zeros(B, dtype=torch.int32))


def _calls():
    def fwd(q, r, kc, vc, sl, out=None, cor=None):
        return plx_decode_fwd(q, r, kc, vc, sl, out)

    def noalloc(q, r, kc, vc, sl, out=None, cor=None):
        return plx_decode_fwd_noalloc(q, r, kc, vc, sl, torch.zeros_like(q) if out is None else out)

    def with_cor(q, r, kc, vc, sl, out=None, cor=None):
        return plx_decode_fwd_cor(q, r, kc, vc, sl, out, cor)

    return {"plx_decode_fwd": fwd, "plx_decode_fwd_noalloc": noalloc,
            "plx_decode_fwd_cor": with_cor}


@pytest.mark.parametrize("call", sorted(_calls()))
@pytest.mark.parametrize("bad,match", [
    ("seqlens", "seqlens"), ("out", "out"), ("r", "r has shape"), ("vcache", "vcache"),
    ("kdim", "kcache"), ("qdim", "q must be"),
])
def test_decode_shape_errors_come_before_any_launch(call, bad, match):
    q, r, kc, vc, sl = _decode_args()
    out = None
    if bad == "seqlens":
        sl = sl[:2]
    elif bad == "out":
        out = torch.zeros(2, 4, 128, dtype=torch.bfloat16)
    elif bad == "r":
        r = r[:, :3]
    elif bad == "vcache":
        vc = vc[:40]
    elif bad == "kdim":
        kc = torch.zeros(50, 2, 64, dtype=torch.bfloat16)
        vc = kc
    elif bad == "qdim":
        q = q[None]
    with pytest.raises(ValueError, match=match):
        _calls()[call](q, r, kc, vc, sl, out=out)


def test_decode_cor_shape_is_checked():
    q, r, kc, vc, sl = _decode_args()
    with pytest.raises(ValueError, match="cor"):
        plx_decode_fwd_cor(q, r, kc, vc, sl, cor=torch.zeros(3, 2))


@pytest.mark.parametrize("call", sorted(_calls()))
def test_decode_host_tensors_are_rejected(call):
    """Right shapes on the host: rejected as not on a CUDA device, still
    before any launch."""
    with pytest.raises(ValueError, match="CUDA"):
        _calls()[call](*_decode_args())
