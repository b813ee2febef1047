"""Pins for the gradient oracle (CPU only).

The oracle differentiates the explicit-Sigma definition with torch.autograd.
These tests tie it to things other than itself: the pinned C oracle for the
forward values, finite differences for the gradient, a library covariance for
the exact rho gradient, the library softmax attention's own gradients at
rho = 0, and two invariants of the definition. The closed-form gradient that
the GPU kernels stream, as the expanded oracle evaluates it densely for
full-size checks, is checked against autograd through the explicit
definition.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import expanded
from oracle import grad as ograd


def _inputs(B, Hq, Hkv, L, d, seed, r_std=0.3):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, L, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, L, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, L, d, generator=g, dtype=torch.float64)
    r = r_std * torch.randn(B, Hq, L, d, generator=g, dtype=torch.float64)
    do = torch.randn(B, Hq, L, d, generator=g, dtype=torch.float64)
    return q, k, v, r, do


def test_forward_matches_the_c_oracle():
    q, k, v, r, _ = _inputs(2, 4, 2, 70, 8, 1)
    o, osa, sbar = ograd.prefill_forward(q, k, v, r)
    ref, _ = oracle.prefill(q, k, v, r)
    np.testing.assert_allclose(o.numpy(), ref, rtol=0, atol=1e-12)


def test_forward_parts_against_library_and_closed_forms():
    """o^SA is torch's fp64 causal softmax attention; sbar is rho . mu with
    the key mean from numpy's weighted average; row 0 gives sbar = rho.k_0."""
    q, k, v, r, _ = _inputs(1, 2, 1, 40, 6, 2)
    _, osa, sbar = ograd.prefill_forward(q, k, v, r)
    kx, vx = (t.repeat_interleave(2, dim=1) for t in (k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(q, kx, vx, is_causal=True)
    np.testing.assert_allclose(osa.numpy(), ref.numpy(), rtol=0, atol=1e-12)
    for h, i in [(0, 0), (1, 7), (0, 39)]:
        w = scipy.special.softmax(kx[0, h, :i + 1].numpy() @ q[0, h, i].numpy() / math.sqrt(6))
        mu = np.average(kx[0, h, :i + 1].numpy(), axis=0, weights=w)
        assert abs(sbar[0, h, i].item() - r[0, h, i].numpy() @ mu) < 1e-12
    assert torch.allclose(sbar[0, :, 0], (r[0, :, 0] * kx[0, :, 0]).sum(-1), rtol=0, atol=1e-13)


def test_gradient_matches_finite_differences():
    q, k, v, r, _ = _inputs(1, 2, 1, 5, 3, 3)
    ins = [t.clone().requires_grad_(True) for t in (q, k, v, r)]
    assert torch.autograd.gradcheck(lambda *a: ograd.forward_parts(*a)[0], ins, eps=1e-6,
                                    atol=1e-8, rtol=1e-6)


def test_rho_gradient_is_minus_sigma_transpose_times_dout():
    """o_i is affine in rho_i with slope -Sigma_i, so dL/drho_i = -Sigma_i^T g_i;
    Sigma_i from numpy's weighted covariance with scipy's softmax weights."""
    B, Hq, Hkv, L, d = 1, 2, 1, 12, 5
    q, k, v, r, do = _inputs(B, Hq, Hkv, L, d, 4)
    _, _, _, dr = ograd.prefill_grad(q, k, v, r, do)
    for h in range(Hq):
        for i in range(L):
            K, V = k[0, 0, :i + 1].numpy(), v[0, 0, :i + 1].numpy()
            w = scipy.special.softmax(K @ q[0, h, i].numpy() / math.sqrt(d))
            sig = (np.zeros((d, d)) if i == 0 else
                   np.cov(np.vstack([V.T, K.T]), aweights=w, bias=True)[:d, d:])
            np.testing.assert_allclose(dr[0, h, i].numpy(), -sig.T @ do[0, h, i].numpy(),
                                       rtol=0, atol=1e-12)


def test_rho_zero_gradients_are_softmax_attention_gradients():
    q, k, v, r, do = _inputs(2, 4, 2, 30, 8, 5)
    dq, dk, dv, _ = ograd.prefill_grad(q, k, v, torch.zeros_like(r), do)
    ins = [t.clone().requires_grad_(True) for t in (q, k, v)]
    o = torch.nn.functional.scaled_dot_product_attention(
        ins[0], ins[1].repeat_interleave(2, dim=1), ins[2].repeat_interleave(2, dim=1),
        is_causal=True)
    ref = torch.autograd.grad(o, ins, grad_outputs=do)
    for got, want in zip((dq, dk, dv), ref):
        np.testing.assert_allclose(got.numpy(), want.numpy(), rtol=0, atol=1e-11)


def test_shift_invariants_of_the_gradients():
    """k_j + c for every j leaves every o unchanged, so the key gradients of a
    kv head sum to zero; v_j + c moves every o by c, so the value gradients
    sum to the output gradients of the heads that read it."""
    q, k, v, r, do = _inputs(2, 4, 2, 33, 8, 6)
    _, dk, dv, _ = ograd.prefill_grad(q, k, v, r, do)
    np.testing.assert_allclose(dk.sum(2).numpy(), 0.0, rtol=0, atol=1e-11)
    want = do.sum(2).reshape(2, 2, 2, 8).sum(2)  # heads 2g, 2g+1 read kv head g
    np.testing.assert_allclose(dv.sum(2).numpy(), want.numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("B,Hq,Hkv,L,d,block", [(1, 2, 1, 17, 4, 17), (2, 4, 2, 40, 8, 9)])
def test_expanded_closed_form_matches_autograd(B, Hq, Hkv, L, d, block):
    """The closed-form gradient of the expanded oracle (dense fp64, query rows
    in blocks) against autograd through the explicit definition."""
    q, k, v, r, do = _inputs(B, Hq, Hkv, L, d, 7 + L)
    want = ograd.prefill_grad(q, k, v, r, do)
    got = expanded.prefill_grad(q, k, v, r, do, row_block=block)
    for name, g_, w_ in zip("qkvr", got, want):
        np.testing.assert_allclose(g_, w_.numpy(), rtol=0, atol=1e-11, err_msg=name)


def test_row_and_key_gradients_match_the_full_gradient():
    """The per-row and per-key walks used at full size agree with the
    whole-tensor gradient on a small case."""
    q, k, v, r, do = _inputs(2, 4, 2, 11, 6, 9)
    dq, dk, dv, dr = ograd.prefill_grad(q, k, v, r, do)
    rows = [(0, 0, 0), (1, 3, 10), (0, 2, 5)]
    gq, gr = ograd.prefill_grad_rows(q, k, v, r, do, rows)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(gq[n].numpy(), dq[b, h, i].numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(gr[n].numpy(), dr[b, h, i].numpy(), rtol=0, atol=1e-12)
    keys = [(0, 1, 10), (1, 0, 8), (1, 1, 0)]
    gk, gv = ograd.prefill_grad_keys(q, k, v, r, do, keys)
    for n, (b, g, j) in enumerate(keys):
        np.testing.assert_allclose(gk[n].numpy(), dk[b, g, j].numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(gv[n].numpy(), dv[b, g, j].numpy(), rtol=0, atol=1e-12)
