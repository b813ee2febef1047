"""Parallax forward oracle (fp64, CPU) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The product
library never calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``plx_oracle.c`` (plain C, fp64): for each query it
forms the softmax weights, the softmax output o^SA, the weighted key mean, the
explicit d x d weighted KV cross-covariance Sigma, and o = o^SA - Sigma rho
(page "Parallax: parametrized local linear attention for language modeling",
section "Core mechanism", output equation). This module compiles that file
with gcc, loads it with ctypes and walks the (batch, head, row) index space:

* ``prefill``: causal -- query i of head h sees keys 0..i of KV head h // G,
  G = Hq / Hkv (consecutive grouping, the plainest GQA reading); with more
  keys than queries the queries are the last positions (a chunk appended to
  a cache) and query i sees keys 0 .. Lk - L + i.
* ``decode``: one query per (sequence, head) sees all ``seqlens[b]`` cached
  keys; the cache is packed ``[sum(seqlens), Hkv, d]``.

With ``with_cor=True`` both also return the correction-to-output ratio
|Sigma rho| / |o| per query (0 where |o| = 0), the COR that the same page
reports in its experimental results; the norms are Euclidean (a reading: the
pages give no formula).

Inputs may be numpy arrays or CPU torch tensors of any float dtype; every
slice is upcast to float64 before the C code sees it, so the oracle works on
exactly the (bf16- or fp32-rounded) values a device kernel receives.

Every function is pinned by ``tests/test_oracle.py`` to things other than
itself: a hand-derived worked example, closed forms, the rho = 0 reduction to
a library softmax attention, a library weighted covariance, a brute-force
dense evaluation of the streaming identity, and invariants of the definition.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "plx_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libplx_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile plx_oracle.c into a shared library with gcc; return its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.plx_oracle_query.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, dp, dp,
                                             dp, ctypes.c_long, dp, ctypes.c_long, dp, dp, dp, dp]
            lib.plx_oracle_query.restype = ctypes.c_int
            lib.plx_oracle_rows.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.c_int,
                                            ctypes.c_double, dp, dp, dp, dp, dp, dp, dp]
            lib.plx_oracle_rows.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Contiguous float64 numpy copy of a numpy array or CPU torch tensor."""
    if not isinstance(x, np.ndarray):
        import torch  # local: the oracle itself needs only numpy
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def query(q, rho, K, V, tau=None, with_sigma=False, with_cor=False):
    """One query vector against all rows of K and V (n x d).

    Returns (o, lse), then Sigma (Sigma[a, c] = value dim a, key dim c) if
    ``with_sigma``, then cor = |Sigma rho| / |o| if ``with_cor``.
    """
    lib = _load()
    q = _f64(q); rho = _f64(rho); K = _f64(K); V = _f64(V)
    n, d = K.shape if K.ndim == 2 else (0, q.shape[0])
    tau = 1.0 / math.sqrt(d) if tau is None else float(tau)
    out = np.empty(d); lse = np.empty(1); cor = np.empty(1)
    sig = np.empty((d, d)) if with_sigma else None
    if n == 0:
        K = np.zeros((1, d)); V = np.zeros((1, d))
    rc = lib.plx_oracle_query(n, d, tau, _ptr(q), _ptr(rho), _ptr(K), d, _ptr(V), d,
                              _ptr(out), _ptr(lse), _ptr(sig) if with_sigma else None,
                              _ptr(cor) if with_cor else None)
    if rc:
        raise MemoryError("oracle allocation failed")
    res = (out, float(lse[0]))
    if with_sigma:
        res += (sig,)
    if with_cor:
        res += (float(cor[0]),)
    return res


def _rows(nkeys, Q, R, K, V, tau):
    lib = _load()
    nkeys = np.ascontiguousarray(nkeys, dtype=np.int32)
    n, d = Q.shape
    out = np.empty((n, d)); lse = np.empty(n); cor = np.empty(n)
    if K.shape[0] == 0:
        K = np.zeros((1, d)); V = np.zeros((1, d))
    rc = lib.plx_oracle_rows(n, nkeys.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), d, tau,
                             _ptr(Q), _ptr(R), _ptr(K), _ptr(V), _ptr(out), _ptr(lse), _ptr(cor))
    if rc:
        raise MemoryError("oracle allocation failed")
    return out, lse, cor


def prefill(q, k, v, r, rows=None, threads=None, with_cor=False):
    """Causal Parallax prefill.

    q, r: [B, Hq, L, d]; k, v: [B, Hkv, Lk, d] with Lk >= L. The L queries are
    the last L of the Lk positions, so query i sees keys 0 .. Lk - L + i
    (Lk == L: ordinary causal prefill; Lk > L: a chunk appended to an existing
    cache). ``rows`` is None (every row) or an iterable of (b, h, i). Returns
    (out, lse), or (out, lse, cor) with ``with_cor``: with rows=None, out is
    [B, Hq, L, d] and lse, cor [B, Hq, L]; otherwise out is [n, d], lse and
    cor [n] in the order of ``rows``.
    """
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    offset = k.shape[2] - L
    assert offset >= 0
    assert Hq % Hkv == 0
    G = Hq // Hkv
    tau = 1.0 / math.sqrt(d)
    if rows is None:
        rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(L)]
        full = True
    else:
        rows = [tuple(int(x) for x in t) for t in rows]
        full = False
    groups = {}
    for n, (b, h, i) in enumerate(rows):
        groups.setdefault((b, h), []).append((n, i))
    out = np.empty((len(rows), d)); lse = np.empty(len(rows)); cor = np.empty(len(rows))

    def work(key):
        b, h = key
        items = groups[key]
        idx = np.array([i for _, i in items])
        Kb = _f64(k[b, h // G]); Vb = _f64(v[b, h // G])
        Qb = _f64(q[b, h])[idx]; Rb = _f64(r[b, h])[idx]
        o, l, c = _rows(offset + idx + 1, Qb, Rb, Kb, Vb, tau)
        for (n, _), on, ln, cn in zip(items, o, l, c):
            out[n] = on; lse[n] = ln; cor[n] = cn

    _parallel(work, list(groups), threads)
    if full:
        out, lse, cor = out.reshape(B, Hq, L, d), lse.reshape(B, Hq, L), cor.reshape(B, Hq, L)
    return (out, lse, cor) if with_cor else (out, lse)


def decode(q, r, kcache, vcache, seqlens, pairs=None, threads=None, with_cor=False):
    """Parallax decode: one query per (sequence b, head h) over its whole cache.

    q, r: [B, Hq, d]; kcache, vcache: packed [sum(seqlens), Hkv, d], sequence b
    at token offset sum(seqlens[:b]). ``pairs`` is None (all) or an iterable of
    (b, h). Returns (out, lse) shaped [B, Hq, d] / [B, Hq] or [n, d] / [n],
    and cor shaped like lse after them with ``with_cor``.
    """
    B, Hq, d = q.shape
    Hkv = kcache.shape[1]
    G = Hq // Hkv
    tau = 1.0 / math.sqrt(d)
    lens = [int(x) for x in (seqlens.tolist() if hasattr(seqlens, "tolist") else seqlens)]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    full = pairs is None
    pairs = [(b, h) for b in range(B) for h in range(Hq)] if full else [tuple(p) for p in pairs]
    out = np.empty((len(pairs), d)); lse = np.empty(len(pairs)); cor = np.empty(len(pairs))

    def work(n):
        b, h = pairs[n]
        lo, hi = int(offs[b]), int(offs[b + 1])
        Kb = _f64(kcache[lo:hi, h // G]); Vb = _f64(vcache[lo:hi, h // G])
        o, l, c = _rows(np.array([hi - lo]), _f64(q[b, h])[None], _f64(r[b, h])[None], Kb, Vb, tau)
        out[n] = o[0]; lse[n] = l[0]; cor[n] = c[0]

    _parallel(work, list(range(len(pairs))), threads)
    if full:
        out, lse, cor = out.reshape(B, Hq, d), lse.reshape(B, Hq), cor.reshape(B, Hq)
    return (out, lse, cor) if with_cor else (out, lse)


def _parallel(fn, items, threads):
    threads = default_threads() if threads is None else threads
    if threads <= 1 or len(items) <= 1:
        for it in items:
            fn(it)
        return
    # ctypes releases the GIL for the duration of each C call, so plain
    # threads give real parallelism here (and are safe next to CUDA).
    with ThreadPoolExecutor(max_workers=min(threads, len(items))) as ex:
        list(ex.map(fn, items))


def qkvr_projection(x, w, B, L, Hq, Hkv, d):
    """The four input projections of a Parallax layer in one product.

    Page "Parallax: parametrized local linear attention for language
    modeling", section "Core mechanism": the probe is rho_i = W_R x_i, a
    linear map of the layer input like q, k and v. x is [B * L, D] (token
    rows, sequence b's tokens at rows b L .. b L + L - 1); w stacks
    [W_Q; W_K; W_V; W_R] as [(2 Hq + 2 Hkv) d, D] rows (output features).
    Returns q, k, v, r as float64 arrays [B, Hq, L, d], [B, Hkv, L, d],
    [B, Hkv, L, d], [B, Hq, L, d]: y = x w^T split at the feature
    boundaries, each part's features grouped into heads of d.
    """
    x = _f64(x)
    w = _f64(w)
    y = x @ w.T  # [B L, F]
    bounds = np.cumsum([0, Hq * d, Hkv * d, Hkv * d, Hq * d])
    outs = []
    for (lo, hi), H in zip(zip(bounds[:-1], bounds[1:]), (Hq, Hkv, Hkv, Hq)):
        outs.append(np.ascontiguousarray(y[:, lo:hi].reshape(B, L, H, d).transpose(0, 2, 1, 3)))
    return tuple(outs)
