"""Thin ctypes binding over libplx.so (argument marshalling only).

Every function here has the name of the C entry point it calls (declared in
include/plx.h) and does nothing but check tensor shapes/dtypes/devices, pass
``data_ptr()`` values and the current CUDA stream, and turn a non-OK status
into an exception. All arithmetic runs in the library's kernels; there is no
fallback: if libplx.so is missing or fails to load, every call raises.
PyTorch supplies device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libplx.so")

PLX_OK = 0
PLX_ERR_INVALID_ARG = 1
PLX_ERR_UNSUPPORTED = 2
PLX_ERR_CUDA = 3
PLX_ERR_DEVICE_TIMEOUT = 4
PLX_ERR_BOUNDS = 5

# Every symbol the header declares, with its ctypes signature.
_vp, _i, _sz, _ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong
SIGNATURES = {
    "plx_prefill_fwd": (_i, [_vp] * 6 + [_i] * 5 + [_vp]),
    "plx_prefill_fwd_f32": (_i, [_vp] * 6 + [_i] * 5 + [_vp]),
    "plx_prefill_fwd_chunk": (_i, [_vp] * 6 + [_i] * 6 + [_vp]),
    "plx_prefill_fwd_cor": (_i, [_vp] * 7 + [_i] * 6 + [_vp]),
    "plx_prefill_fwd_train": (_i, [_vp] * 8 + [_i] * 5 + [_vp]),
    "plx_prefill_bwd": (_i, [_vp] * 13 + [_i] * 5 + [_vp]),
    "plx_qkvr_proj": (_i, [_vp] * 6 + [_i] * 6 + [_vp]),
    "plx_decode_fwd": (_i, [_vp] * 6 + [_i] * 4 + [_vp]),
    "plx_decode_fwd_ex": (_i, [_vp] * 6 + [_i] * 5 + [_vp, _sz, _vp]),
    "plx_decode_fwd_noalloc": (_i, [_vp] * 6 + [_i] * 4 + [_vp]),
    "plx_decode_fwd_cor": (_i, [_vp] * 7 + [_i] * 4 + [_vp]),
    "plx_decode_workspace_bytes": (_sz, [_i] * 5),
    "plx_decode_default_nsplit": (_i, [_i] * 2),
    "plx_check_device_error": (_i, [_vp]),
    "plx_debug_timeout_probe": (_i, [_ll, _vp]),
    "plx_status_string": (ctypes.c_char_p, [_i]),
    "plx_last_error_message": (ctypes.c_char_p, []),
}


class PlxError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


_lib = None
_lock = threading.Lock()


def lib():
    """Load libplx.so (built by ``build.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libplx.so not built ({LIB_PATH}); run "
                    "python -m parametrized_local_linear_gb300.build")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def load_debug_lib():
    """libplx_debug.so, the build with device-side bounds checks (see
    include/plx.h), loaded with the same signatures; built if missing."""
    from . import build
    L = ctypes.CDLL(build.build(debug_bounds=True))
    for name, (res, args) in SIGNATURES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


def _check(status: int):
    if status != PLX_OK:
        msg = lib().plx_last_error_message().decode(errors="replace")
        raise PlxError(status, msg or lib().plx_status_string(status).decode())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, ndim, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _prefill(fn, dtype, q, k, v, r, out, lse, stream):
    _need(q, "q", dtype, 4)
    dev = q.device
    for name, t in (("k", k), ("v", v), ("r", r)):
        _need(t, name, dtype, 4, dev)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    if tuple(r.shape) != tuple(q.shape):
        raise ValueError("r must have the shape of q")
    if tuple(k.shape) != (B, Hkv, L, d) or tuple(v.shape) != (B, Hkv, L, d):
        raise ValueError("k and v must be [B, Hkv, L, d] matching q")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dtype, 4, dev)
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have the shape of q")
    if lse is not None:
        _need(lse, "lse", torch.float32, 3, dev)
        if tuple(lse.shape) != (B, Hq, L):
            raise ValueError("lse must be [B, Hq, L]")
    with torch.cuda.device(dev):
        st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), r.data_ptr(), out.data_ptr(),
                lse.data_ptr() if lse is not None else None, B, Hq, Hkv, L, d,
                _stream(stream, dev))
    _check(st)
    return out, lse


def plx_prefill_fwd(q, k, v, r, out=None, lse=None, stream=None):
    """Causal Parallax prefill, bf16 (see include/plx.h). Returns (out, lse)."""
    return _prefill(lib().plx_prefill_fwd, torch.bfloat16, q, k, v, r, out, lse, stream)


def plx_prefill_fwd_chunk(q, k, v, r, out=None, lse=None, stream=None):
    """Chunked causal prefill (see include/plx.h): q, r [B, Hq, Lq, d] are the
    last Lq positions of k, v [B, Hkv, Lk, d]. Returns (out, lse)."""
    out, lse, _ = _prefill_chunk(q, k, v, r, out, lse, None, stream)
    return out, lse


def plx_prefill_fwd_cor(q, k, v, r, out=None, lse=None, cor=None, stream=None):
    """Chunked causal prefill that also writes the correction-to-output ratio
    |Sigma rho| / |o| per row (see include/plx.h). ``cor`` is fp32
    [B, Hq, Lq] (allocated if None). Returns (out, lse, cor)."""
    if cor is None:
        cor = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    return _prefill_chunk(q, k, v, r, out, lse, cor, stream)


def _prefill_chunk(q, k, v, r, out, lse, cor, stream):
    _need(q, "q", torch.bfloat16, 4)
    dev = q.device
    for name, t in (("k", k), ("v", v), ("r", r)):
        _need(t, name, torch.bfloat16, 4, dev)
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if tuple(r.shape) != tuple(q.shape):
        raise ValueError("r must have the shape of q")
    if tuple(k.shape) != (B, Hkv, Lk, d) or tuple(v.shape) != (B, Hkv, Lk, d):
        raise ValueError("k and v must be [B, Hkv, Lk, d] matching q")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 4, dev)
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have the shape of q")
    for name, t in (("lse", lse), ("cor", cor)):
        if t is not None:
            _need(t, name, torch.float32, 3, dev)
            if tuple(t.shape) != (B, Hq, Lq):
                raise ValueError(f"{name} must be [B, Hq, Lq]")
    lse_ptr = lse.data_ptr() if lse is not None else None
    with torch.cuda.device(dev):
        if cor is None:
            st = lib().plx_prefill_fwd_chunk(q.data_ptr(), k.data_ptr(), v.data_ptr(), r.data_ptr(),
                                             out.data_ptr(), lse_ptr, B, Hq, Hkv, Lq, Lk, d,
                                             _stream(stream, dev))
        else:
            st = lib().plx_prefill_fwd_cor(q.data_ptr(), k.data_ptr(), v.data_ptr(), r.data_ptr(),
                                           out.data_ptr(), lse_ptr, cor.data_ptr(), B, Hq, Hkv, Lq,
                                           Lk, d, _stream(stream, dev))
    _check(st)
    return out, lse, cor


def plx_prefill_fwd_train(q, k, v, r, out=None, lse=None, o1=None, sbar=None, stream=None):
    """Training forward (see include/plx.h): returns (out, lse, o1, sbar), the
    last three being what plx_prefill_bwd needs."""
    _need(q, "q", torch.bfloat16, 4)
    dev = q.device
    for name, t in (("k", k), ("v", v), ("r", r)):
        _need(t, name, torch.bfloat16, 4, dev)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    if tuple(r.shape) != tuple(q.shape) or tuple(k.shape) != (B, Hkv, L, d) or v.shape != k.shape:
        raise ValueError("r must match q; k and v must be [B, Hkv, L, d]")
    out = torch.empty_like(q) if out is None else out
    o1 = torch.empty_like(q) if o1 is None else o1
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=dev) if lse is None else lse
    sbar = torch.empty((B, Hq, L), dtype=torch.float32, device=dev) if sbar is None else sbar
    for name, t in (("out", out), ("o1", o1)):
        _need(t, name, torch.bfloat16, 4, dev)
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} must have the shape of q")
    for name, t in (("lse", lse), ("sbar", sbar)):
        _need(t, name, torch.float32, 3, dev)
        if tuple(t.shape) != (B, Hq, L):
            raise ValueError(f"{name} must be [B, Hq, L]")
    with torch.cuda.device(dev):
        st = lib().plx_prefill_fwd_train(q.data_ptr(), k.data_ptr(), v.data_ptr(), r.data_ptr(),
                                         out.data_ptr(), lse.data_ptr(), o1.data_ptr(),
                                         sbar.data_ptr(), B, Hq, Hkv, L, d, _stream(stream, dev))
    _check(st)
    return out, lse, o1, sbar


def plx_prefill_bwd(q, k, v, r, out, o1, lse, sbar, dout, dq=None, dk=None, dv=None, dr=None,
                    stream=None):
    """Backward of the causal prefill (see include/plx.h). Returns
    (dq, dk, dv, dr), bf16, shaped like q, k, v, r."""
    _need(q, "q", torch.bfloat16, 4)
    dev = q.device
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    for name, t in (("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 4, dev)
        if tuple(t.shape) != (B, Hkv, L, d):
            raise ValueError(f"{name} must be [B, Hkv, L, d]")
    dq = torch.empty_like(q) if dq is None else dq
    dr = torch.empty_like(q) if dr is None else dr
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, like in (("r", r, q), ("out", out, q), ("o1", o1, q), ("dout", dout, q),
                          ("dq", dq, q), ("dr", dr, q), ("dk", dk, k), ("dv", dv, k)):
        _need(t, name, torch.bfloat16, 4, dev)
        if tuple(t.shape) != tuple(like.shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(like.shape)}")
    for name, t in (("lse", lse), ("sbar", sbar)):
        _need(t, name, torch.float32, 3, dev)
        if tuple(t.shape) != (B, Hq, L):
            raise ValueError(f"{name} must be [B, Hq, L]")
    with torch.cuda.device(dev):
        st = lib().plx_prefill_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), r.data_ptr(),
                                   out.data_ptr(), o1.data_ptr(), lse.data_ptr(), sbar.data_ptr(),
                                   dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                   dr.data_ptr(), B, Hq, Hkv, L, d, _stream(stream, dev))
    _check(st)
    return dq, dk, dv, dr


def plx_qkvr_proj(x, w, B, L, Hq, Hkv, d=128, q=None, k=None, v=None, r=None, stream=None):
    """Fused [W_Q; W_K; W_V; W_R] x projection (see include/plx.h): x bf16
    [B * L, D], w bf16 [(2 Hq + 2 Hkv) d, D]. Returns (q, k, v, r) in the
    attention layouts [B, H, L, d]."""
    _need(x, "x", torch.bfloat16, 2)
    dev = x.device
    _need(w, "w", torch.bfloat16, 2, dev)
    T, D = x.shape
    if T != B * L or tuple(w.shape) != ((2 * Hq + 2 * Hkv) * d, D):
        raise ValueError("x must be [B * L, D] and w [(2 Hq + 2 Hkv) d, D]")
    shapes = {"q": (B, Hq, L, d), "k": (B, Hkv, L, d), "v": (B, Hkv, L, d), "r": (B, Hq, L, d)}
    outs = {}
    for name, t in (("q", q), ("k", k), ("v", v), ("r", r)):
        if t is None:
            t = torch.empty(shapes[name], dtype=torch.bfloat16, device=dev)
        _need(t, name, torch.bfloat16, 4, dev)
        if tuple(t.shape) != shapes[name]:
            raise ValueError(f"{name} must be {shapes[name]}")
        outs[name] = t
    with torch.cuda.device(dev):
        st = lib().plx_qkvr_proj(x.data_ptr(), w.data_ptr(), outs["q"].data_ptr(),
                                 outs["k"].data_ptr(), outs["v"].data_ptr(), outs["r"].data_ptr(),
                                 B, L, D, Hq, Hkv, d, _stream(stream, dev))
    _check(st)
    return outs["q"], outs["k"], outs["v"], outs["r"]


def plx_prefill_fwd_f32(q, k, v, r, out=None, lse=None, stream=None):
    """Causal Parallax prefill, fp32 (see include/plx.h). Returns (out, lse)."""
    return _prefill(lib().plx_prefill_fwd_f32, torch.float32, q, k, v, r, out, lse, stream)


def _decode_shapes(q, r, kcache, vcache, seqlens, out=None, cor=None):
    """Shape checks shared by every decode call, made before any device check
    or launch: a short ``seqlens``, ``out`` or ``cor`` would otherwise let the
    kernels read or write past the end of a buffer."""
    if q.dim() != 3:
        raise ValueError(f"q must be [B, Hq, d], got shape {tuple(q.shape)}")
    B, Hq, d = q.shape
    if tuple(r.shape) != tuple(q.shape):
        raise ValueError(f"r has shape {tuple(r.shape)}, expected the shape of q {tuple(q.shape)}")
    if kcache.dim() != 3 or kcache.shape[2] != d:
        raise ValueError(f"kcache must be [T, Hkv, {d}], got shape {tuple(kcache.shape)}")
    if tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError(f"vcache has shape {tuple(vcache.shape)}, expected the shape of kcache "
                         f"{tuple(kcache.shape)}")
    if seqlens.dim() != 1 or seqlens.shape[0] != B:
        raise ValueError(f"seqlens must have shape ({B},), got {tuple(seqlens.shape)}")
    if out is not None and tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out has shape {tuple(out.shape)}, expected the shape of q {tuple(q.shape)}")
    if cor is not None and tuple(cor.shape) != (B, Hq):
        raise ValueError(f"cor has shape {tuple(cor.shape)}, expected ({B}, {Hq})")


def _decode_tensors(q, r, kcache, vcache, seqlens, out, cor=None):
    _decode_shapes(q, r, kcache, vcache, seqlens, out, cor)
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    for name, t in (("r", r), ("kcache", kcache), ("vcache", vcache)):
        _need(t, name, torch.bfloat16, 3, dev)
    _need(seqlens, "seqlens", torch.int32, 1, dev)
    if out is not None:
        _need(out, "out", torch.bfloat16, 3, dev)
    if cor is not None:
        _need(cor, "cor", torch.float32, 2, dev)
    return dev


def plx_decode_fwd(q, r, kcache, vcache, seqlens, out=None, nsplit=0, workspace=None,
                   stream=None):
    """Parallax decode over a packed ragged KV cache (see include/plx.h).

    q, r: bf16 [B, Hq, d]; kcache, vcache: bf16 [sum(seqlens), Hkv, d];
    seqlens: int32 [B] on the device. ``nsplit``/``workspace`` select
    plx_decode_fwd_ex; the defaults call plx_decode_fwd. Returns out.
    """
    dev = _decode_tensors(q, r, kcache, vcache, seqlens, out)
    B, Hq, d = q.shape
    Hkv = kcache.shape[1]
    if out is None:
        out = torch.empty_like(q)
    L = lib()
    with torch.cuda.device(dev):
        s = _stream(stream, dev)
        if nsplit == 0 and workspace is None:
            st = L.plx_decode_fwd(q.data_ptr(), r.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                  seqlens.data_ptr(), out.data_ptr(), B, Hq, Hkv, d, s)
        else:
            ws_ptr, ws_bytes = None, 0
            if workspace is not None:
                if not workspace.is_cuda or workspace.device != dev:
                    raise ValueError("workspace must be on the device of q")
                ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
            st = L.plx_decode_fwd_ex(q.data_ptr(), r.data_ptr(), kcache.data_ptr(),
                                     vcache.data_ptr(), seqlens.data_ptr(), out.data_ptr(), B, Hq,
                                     Hkv, d, int(nsplit), ws_ptr, ws_bytes, s)
    _check(st)
    return out


def plx_decode_fwd_noalloc(q, r, kcache, vcache, seqlens, out, stream=None):
    """Decode through the entry point that allocates nothing (see include/plx.h):
    the partial records go to the library's fixed device array. ``out`` must be
    given (bf16 [B, Hq, d]); returns it."""
    if out is None:
        raise ValueError("out must be given: this entry point allocates nothing")
    dev = _decode_tensors(q, r, kcache, vcache, seqlens, out)
    B, Hq, d = q.shape
    with torch.cuda.device(dev):
        st = lib().plx_decode_fwd_noalloc(q.data_ptr(), r.data_ptr(), kcache.data_ptr(),
                                          vcache.data_ptr(), seqlens.data_ptr(), out.data_ptr(),
                                          B, Hq, kcache.shape[1], d, _stream(stream, dev))
    _check(st)
    return out


def plx_decode_fwd_cor(q, r, kcache, vcache, seqlens, out=None, cor=None, stream=None):
    """Decode that also writes the correction-to-output ratio |Sigma rho| / |o|
    per (sequence, head) (see include/plx.h). ``cor`` is fp32 [B, Hq]
    (allocated if None). Returns (out, cor)."""
    dev = _decode_tensors(q, r, kcache, vcache, seqlens, out, cor)
    B, Hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if cor is None:
        cor = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib().plx_decode_fwd_cor(q.data_ptr(), r.data_ptr(), kcache.data_ptr(),
                                      vcache.data_ptr(), seqlens.data_ptr(), out.data_ptr(),
                                      cor.data_ptr(), B, Hq, kcache.shape[1], d,
                                      _stream(stream, dev))
    _check(st)
    return out, cor


def plx_decode_workspace_bytes(B, Hq, Hkv, d, nsplit) -> int:
    return int(lib().plx_decode_workspace_bytes(B, Hq, Hkv, d, nsplit))


def plx_decode_default_nsplit(B, Hkv) -> int:
    return int(lib().plx_decode_default_nsplit(B, Hkv))


def plx_check_device_error(stream=None, device=None):
    """Synchronise the stream and raise PlxError if a bounded wait ran out."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        _check(lib().plx_check_device_error(_stream(stream, dev)))


def plx_debug_timeout_probe(limit_cycles=100000, stream=None):
    dev = torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        _check(lib().plx_debug_timeout_probe(int(limit_cycles), _stream(stream, dev)))
