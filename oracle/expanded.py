"""Expanded-form Parallax forward and gradient (fp64, CPU) -- TEST
INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this module. It shares no
code with the CUDA path.

The explicit oracle in ``plx_oracle.c`` forms the d x d covariance of every
query, which is too slow for every row of a model-sized workload. This module
evaluates the same output through the identity the streaming algorithm rests
on (page "Parallax: parametrized local linear attention for language
modeling", section "Core mechanism" for the output equation, section
"Hardware-aware algorithm" for the streaming form): with P the softmax
weights of the causal window, T = R K^T the probe-key products (unscaled),
l = rowsum(P),

    O1 = P V / l,   O2 = (P o T) V / l,   s = rowsum(P o T) / l,
    o  = O1 - O2 + O1 * s,   lse = max + ln l,

so that the correction Sigma rho is O2 - O1 * s. It holds exactly because the
weighted mean of v_j - o^SA is zero, which drops the key-mean term of the
covariance. The gradient is the closed form of the same definition (the pages
print no backward pass): with w = P / l, t = T, sbar = s, c = 1 + sbar - t,
u = dout V^T, a = dout . o^SA and D = dout . o + a sbar,

    dt = w (a - u),   ds = w (c u + a t - D),
    dq = tau ds K,   drho = dt K,
    dK = tau ds^T Q + dt^T R,   dV = (w c)^T dout,

dK and dV summed over the query heads that read the kv head.

Everything is dense fp64 matrices and library matrix products on the CPU:
per (batch, head), the scores of a block of query rows against every key
those rows may see, masked, exponentiated against the row max, and multiplied
out. Query rows are independent, so taking them in blocks only bounds memory;
it does not change what a row computes (the key gradients add the blocks'
contributions). Nothing is streamed or rescaled online.

``tests/test_oracle.py`` and ``tests/test_oracle_grad.py`` pin these
functions to the explicit oracle and to autograd through the explicit
definition (and so to everything those are pinned to) on small inputs.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def _f64(x) -> torch.Tensor:
    if isinstance(x, np.ndarray):
        x = torch.from_numpy(x)
    return x.detach().to("cpu", torch.float64)


def _weights(Q, K, tau, nkeys):
    """Normalised causal softmax weights w [n, nk] of query rows Q against the
    keys K (row i sees keys 0 .. nkeys[i] - 1), the row max m and the
    normaliser l (lse = m + ln l)."""
    nk = K.shape[0]
    S = (Q @ K.T) * tau
    S = S.masked_fill(torch.arange(nk)[None, :] >= nkeys[:, None], -math.inf)
    m = S.max(dim=1, keepdim=True).values
    m = torch.where(torch.isfinite(m), m, torch.zeros_like(m))
    P = torch.exp(S - m)
    ell = P.sum(dim=1, keepdim=True)
    w = P / torch.where(ell > 0, ell, torch.ones_like(ell))
    return w, m, ell


def _rows(Q, R, K, V, tau, nkeys):
    """Expanded form for query rows Q, R [n, d], row i seeing keys
    0 .. nkeys[i] - 1 of K, V. Returns (o, lse, o^SA, sbar, correction); a
    row that sees no key gets zeros and lse = -inf."""
    n, d = Q.shape
    nk = int(nkeys.max()) if n else 0
    if nk == 0:
        z = torch.zeros_like(Q)
        return z, torch.full((n,), -math.inf, dtype=torch.float64), z, torch.zeros(n, dtype=torch.float64), z
    K = K[:nk]
    V = V[:nk]
    w, m, ell = _weights(Q, K, tau, nkeys)
    T = R @ K.T
    PT = w * T
    O1 = w @ V
    O2 = PT @ V
    s = PT.sum(dim=1, keepdim=True)
    corr = O2 - O1 * s
    o = O1 - corr
    lse = (m + torch.log(ell)).squeeze(1)
    return o, lse, O1, s.squeeze(1), corr


def _cor(o, corr):
    """|correction| / |o| per row (0 where |o| = 0)."""
    on = np.linalg.norm(o, axis=-1)
    cn = np.linalg.norm(corr, axis=-1)
    return np.where(on > 0, cn / np.where(on > 0, on, 1.0), 0.0)


def prefill(q, k, v, r, row_block=1024, with_parts=False):
    """Causal prefill by the expanded form.

    q, r: [B, Hq, L, d]; k, v: [B, Hkv, Lk, d] with Lk >= L; the L queries are
    the last L positions, so query i sees keys 0 .. Lk - L + i (Lk == L: plain
    causal prefill). Query head h reads KV head h // (Hq / Hkv). Returns
    (out [B, Hq, L, d], lse [B, Hq, L]) as float64 numpy arrays; with
    ``with_parts`` also o^SA [B, Hq, L, d], sbar [B, Hq, L] and the
    correction-to-output ratio cor = |Sigma rho| / |o| [B, Hq, L].
    """
    B, Hq, L, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    assert Lk >= L and Hq % Hkv == 0
    G = Hq // Hkv
    offset = Lk - L
    tau = 1.0 / math.sqrt(d)
    out = np.empty((B, Hq, L, d))
    lse = np.empty((B, Hq, L))
    if with_parts:
        osa = np.empty((B, Hq, L, d))
        sbar = np.empty((B, Hq, L))
        cor = np.empty((B, Hq, L))
    for b in range(B):
        for g in range(Hkv):
            K = _f64(k[b, g])
            V = _f64(v[b, g])
            for h in range(g * G, (g + 1) * G):
                Q = _f64(q[b, h])
                R = _f64(r[b, h])
                for i0 in range(0, L, row_block):
                    i1 = min(L, i0 + row_block)
                    nkeys = offset + torch.arange(i0, i1) + 1
                    o, l, o1, s, corr = _rows(Q[i0:i1], R[i0:i1], K, V, tau, nkeys)
                    out[b, h, i0:i1] = o.numpy()
                    lse[b, h, i0:i1] = l.numpy()
                    if with_parts:
                        osa[b, h, i0:i1] = o1.numpy()
                        sbar[b, h, i0:i1] = s.numpy()
                        cor[b, h, i0:i1] = _cor(o.numpy(), corr.numpy())
    if with_parts:
        return out, lse, osa, sbar, cor
    return out, lse


def decode(q, r, kcache, vcache, seqlens, with_cor=False):
    """Decode by the expanded form: query (b, h) sees all seqlens[b] keys of
    sequence b, stored packed at token offset sum(seqlens[:b]) of
    kcache, vcache [sum(seqlens), Hkv, d]. Returns (out [B, Hq, d],
    lse [B, Hq]) as float64 numpy arrays, and cor [B, Hq] after them with
    ``with_cor``; an empty sequence gives o = 0 and cor = 0."""
    B, Hq, d = q.shape
    Hkv = kcache.shape[1]
    G = Hq // Hkv
    tau = 1.0 / math.sqrt(d)
    lens = [int(x) for x in (seqlens.tolist() if hasattr(seqlens, "tolist") else seqlens)]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    out = np.empty((B, Hq, d))
    lse = np.empty((B, Hq))
    cor = np.empty((B, Hq))
    for b in range(B):
        lo, hi = int(offs[b]), int(offs[b + 1])
        for g in range(Hkv):
            K = _f64(kcache[lo:hi, g])
            V = _f64(vcache[lo:hi, g])
            hs = slice(g * G, (g + 1) * G)
            nkeys = torch.full((G,), hi - lo, dtype=torch.int64)
            o, l, _, _, corr = _rows(_f64(q[b, hs]), _f64(r[b, hs]), K, V, tau, nkeys)
            out[b, hs] = o.numpy()
            lse[b, hs] = l.numpy()
            cor[b, hs] = _cor(o.numpy(), corr.numpy())
    return (out, lse, cor) if with_cor else (out, lse)


def prefill_grad(q, k, v, r, dout, row_block=1024):
    """Gradients (dq, dk, dv, dr) of sum(dout * o) for the causal prefill
    (Lq = Lk = L), by the closed form above, as float64 numpy arrays shaped
    like q, k, v, r."""
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    tau = 1.0 / math.sqrt(d)
    dq = np.empty((B, Hq, L, d))
    dr = np.empty((B, Hq, L, d))
    dk = np.zeros((B, Hkv, L, d))
    dv = np.zeros((B, Hkv, L, d))
    for b in range(B):
        for g in range(Hkv):
            K = _f64(k[b, g])
            V = _f64(v[b, g])
            dK = torch.zeros(L, d, dtype=torch.float64)
            dV = torch.zeros(L, d, dtype=torch.float64)
            for h in range(g * G, (g + 1) * G):
                Q = _f64(q[b, h])
                R = _f64(r[b, h])
                dO = _f64(dout[b, h])
                for i0 in range(0, L, row_block):
                    i1 = min(L, i0 + row_block)
                    nkeys = torch.arange(i0, i1) + 1
                    Kb, Vb = K[:i1], V[:i1]
                    Qb, Rb, gb = Q[i0:i1], R[i0:i1], dO[i0:i1]
                    w, _, _ = _weights(Qb, Kb, tau, nkeys)
                    t = Rb @ Kb.T
                    sb = (w * t).sum(dim=1, keepdim=True)
                    c = 1.0 + sb - t
                    osa = w @ Vb
                    o = (w * c) @ Vb
                    u = gb @ Vb.T
                    a = (gb * osa).sum(dim=1, keepdim=True)
                    D = (gb * o).sum(dim=1, keepdim=True) + a * sb
                    dt = w * (a - u)
                    ds = w * (c * u + a * t - D)
                    dq[b, h, i0:i1] = (tau * ds @ Kb).numpy()
                    dr[b, h, i0:i1] = (dt @ Kb).numpy()
                    dK[:i1] += tau * ds.T @ Qb + dt.T @ Rb
                    dV[:i1] += (w * c).T @ gb
            dk[b, g] = dK.numpy()
            dv[b, g] = dV.numpy()
    return dq, dk, dv, dr
