"""Gradients of the causal Parallax forward (fp64, CPU) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and the CPU legs of ``bench.py`` may import this module; the
product library never calls it and shares no code with it.

The pages ("Parallax: parametrized local linear attention for language
modeling", section "Core mechanism", output equation; section "Experimental
results" for the training runs) print no backward pass. The gradient of the
method is the gradient of its forward definition, so this module writes that
definition out in plain torch fp64 -- scores, softmax weights, o^SA, the key
mean, the explicit d x d weighted cross-covariance Sigma per query, and
o = o^SA - Sigma rho -- and lets torch.autograd differentiate it. Nothing is
fused or reordered beyond forming Sigma for a block of query rows at a time
(to bound memory); no streaming identity and no hand-derived gradient appear.

Conventions as in the rest of the oracle: q, r [B, Hq, L, d]; k, v
[B, Hkv, L, d]; query head h reads kv head h // (Hq / Hkv); causal window
j <= i with the diagonal; tau = 1 / sqrt(d); rho is r.
"""
from __future__ import annotations

import math

import torch

_ROWS = 64  # query rows per block of explicit Sigma matrices


def _f64(x) -> torch.Tensor:
    if not isinstance(x, torch.Tensor):
        x = torch.as_tensor(x)
    return x.detach().to("cpu", torch.float64)


def forward_parts(q, k, v, r):
    """The explicit definition, differentiably. Returns (o, osa, sbar):
    o = o^SA - Sigma rho, o^SA the softmax attention output, and
    sbar = sum_j w_j (rho . k_j), the softmax-weighted mean of rho . k (the
    key-side mean of the correction's probe projection)."""
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    kx = k.repeat_interleave(G, dim=1)
    vx = v.repeat_interleave(G, dim=1)
    tau = 1.0 / math.sqrt(d)
    scores = tau * (q @ kx.transpose(-1, -2))
    causal = torch.ones(L, L, dtype=torch.bool).tril()
    w = torch.softmax(scores.masked_fill(~causal, -math.inf), dim=-1)  # [B, Hq, L, L]
    osa = w @ vx
    mu = w @ kx
    corr = []
    for i0 in range(0, L, _ROWS):
        i1 = min(L, i0 + _ROWS)
        vc = vx[:, :, None, :, :] - osa[:, :, i0:i1, None, :]   # [B, Hq, rows, L, d]
        kc = kx[:, :, None, :, :] - mu[:, :, i0:i1, None, :]
        wb = w[:, :, i0:i1, :, None]
        sigma = (wb * vc).transpose(-1, -2) @ kc                  # [B, Hq, rows, d, d]
        corr.append((sigma @ r[:, :, i0:i1, :, None]).squeeze(-1))
    o = osa - torch.cat(corr, dim=2)
    sbar = (w * (r @ kx.transpose(-1, -2))).sum(-1)
    return o, osa, sbar


def prefill_forward(q, k, v, r):
    """(o, osa, sbar) in fp64 without gradients."""
    with torch.no_grad():
        return forward_parts(*(_f64(t) for t in (q, k, v, r)))


def prefill_grad(q, k, v, r, dout):
    """Gradients (dq, dk, dv, dr) of sum(dout * o) with o the causal Parallax
    forward, by autograd through the explicit definition, in fp64."""
    ins = [_f64(t).requires_grad_(True) for t in (q, k, v, r)]
    with torch.enable_grad():
        o, _, _ = forward_parts(*ins)
        grads = torch.autograd.grad(o, ins, grad_outputs=_f64(dout))
    return tuple(g.detach() for g in grads)


def _row_output(q, r, K, V):
    """o for one query (q, r: [d]) over keys K, V ([n, d]), explicit Sigma."""
    d = q.shape[0]
    w = torch.softmax((K @ q) / math.sqrt(d), dim=0)
    osa = w @ V
    mu = w @ K
    sigma = ((V - osa) * w[:, None]).transpose(0, 1) @ (K - mu)
    return osa - sigma @ r


def row_grads(q, r, K, V, g):
    """Gradients of g . o for one query row over its keys: (dq, dr, dK, dV)
    with dK, dV [n, d], by autograd through the explicit definition."""
    ins = [_f64(t).requires_grad_(True) for t in (q, r, K, V)]
    with torch.enable_grad():
        o = _row_output(*ins)
        dq, dr, dK, dV = torch.autograd.grad(o, ins, grad_outputs=_f64(g))
    return dq, dr, dK, dV


def prefill_grad_rows(q, k, v, r, dout, rows):
    """dq and dr of the listed query rows (b, h, i) of a causal prefill: row i
    depends on nothing but its own forward, so each is one row's gradient.
    Returns two [n, d] tensors in the order of ``rows``."""
    G = q.shape[1] // k.shape[1]
    dq, dr = [], []
    for b, h, i in rows:
        gq, gr, _, _ = row_grads(q[b, h, i], r[b, h, i], k[b, h // G, :i + 1], v[b, h // G, :i + 1],
                                 dout[b, h, i])
        dq.append(gq)
        dr.append(gr)
    return torch.stack(dq), torch.stack(dr)


def prefill_grad_keys(q, k, v, r, dout, keys):
    """dk and dv of the listed keys (b, kv head, j): the sum, over every query
    head of the group and every row i >= j, of that row's key gradient. Cheap
    for keys near the end of the sequence. Returns two [n, d] tensors."""
    B, Hq, L, d = q.shape
    G = Hq // k.shape[1]
    dk, dv = [], []
    for b, g, j in keys:
        ak = torch.zeros(d, dtype=torch.float64)
        av = torch.zeros(d, dtype=torch.float64)
        for h in range(g * G, (g + 1) * G):
            for i in range(j, L):
                _, _, gK, gV = row_grads(q[b, h, i], r[b, h, i], k[b, g, :i + 1], v[b, g, :i + 1],
                                         dout[b, h, i])
                ak += gK[j]
                av += gV[j]
        dk.append(ak)
        dv.append(av)
    return torch.stack(dk), torch.stack(dv)
