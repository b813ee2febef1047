"""GPU backward of the causal prefill (and the training forward it needs)
against the fp64 gradient oracle (autograd through the explicit-Sigma
definition)."""
import numpy as np
import pytest
import torch

from oracle import grad as ograd
from parametrized_local_linear_gb300 import (inputs, plx_check_device_error, plx_prefill_bwd,
                                             plx_prefill_fwd, plx_prefill_fwd_train)

from helpers import SBAR_ABS, assert_bf16_close, assert_grad_close, device, sample_rows

pytestmark = pytest.mark.gpu


def _case(B, Hq, Hkv, L, seed):
    q, k, v, r = inputs.prefill_inputs(B, Hq, Hkv, L, 128, torch.bfloat16, 0.05, seed)
    g = torch.Generator().manual_seed(seed + 7)
    do = torch.randn(B, Hq, L, 128, generator=g).to(torch.bfloat16)
    return q, k, v, r, do


def _gpu_grads(q, k, v, r, do):
    dev = device()
    qd, kd, vd, rd, dod = (t.to(dev) for t in (q, k, v, r, do))
    out, lse, o1, sbar = plx_prefill_fwd_train(qd, kd, vd, rd)
    fill = lambda t: torch.full_like(t, float("nan"))  # noqa: E731
    grads = plx_prefill_bwd(qd, kd, vd, rd, out, o1, lse, sbar, dod,
                            fill(qd), fill(kd), fill(vd), fill(rd))
    plx_check_device_error()
    return [g.double().cpu() for g in grads]


def test_train_forward_saves_osa_and_sbar():
    dev = device()
    q, k, v, r, _ = _case(1, 4, 2, 300, 41)
    qd, kd, vd, rd = (t.to(dev) for t in (q, k, v, r))
    out, lse, o1, sbar = plx_prefill_fwd_train(qd, kd, vd, rd)
    plain, plain_lse = plx_prefill_fwd(qd, kd, vd, rd, lse=torch.empty_like(lse))
    plx_check_device_error()
    assert torch.equal(out, plain) and torch.equal(lse, plain_lse)
    _, osa, ref_sbar = ograd.prefill_forward(q, k, v, r)
    assert_bf16_close(o1.double().cpu().numpy(), osa.numpy(), "o^SA")
    # sbar comes from fp32 scores and probe products (no bf16 rounding).
    np.testing.assert_allclose(sbar.double().cpu().numpy(), ref_sbar.numpy(), rtol=0, atol=SBAR_ABS)


@pytest.mark.parametrize("B,Hq,Hkv,L", [
    (1, 2, 1, 1),      # one token: Sigma = 0, the softmax has one weight
    (2, 2, 1, 2),      # two tokens
    (1, 2, 1, 65),     # one key block, a 1-row second query tile
    (1, 2, 1, 200),    # ragged last query and key tiles
    (2, 4, 2, 130),    # GQA pairs, just over one 128-row block
    (1, 2, 2, 64),     # one key tile, no GQA
    (1, 4, 1, 257),    # a group of 4 query heads per kv head; 1-row tail
    (1, 8, 1, 150),    # a group of 8: the key-block kernel walks 8 heads
    (1, 16, 1, 70),    # one kv head for 16 query heads (MQA)
])
def test_backward_matches_oracle(B, Hq, Hkv, L):
    q, k, v, r, do = _case(B, Hq, Hkv, L, 50 + L)
    got = _gpu_grads(q, k, v, r, do)
    want = ograd.prefill_grad(q, k, v, r, do)
    # With one or two keys per row the exact score and probe gradients vanish
    # or nearly so (one key: dq = dk = drho = 0, dv = dout), while the kernel
    # carries the forward's bf16 rounding of P o T (O2 uses the rounded
    # product, sigma the fp32 one). There the error is measured against the
    # largest gradient of the step instead of each tensor's own largest.
    scale = max(float(w_.abs().max()) for w_ in want) if L <= 2 else None
    for name, g_, w_ in zip(("dq", "dk", "dv", "dr"), got, want):
        assert_grad_close(g_.numpy(), w_.numpy(), f"{name} B{B} Hq{Hq} Hkv{Hkv} L{L}", scale=scale)


def test_backward_is_deterministic():
    q, k, v, r, do = _case(1, 2, 1, 333, 61)
    a = _gpu_grads(q, k, v, r, do)
    b = _gpu_grads(q, k, v, r, do)
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_backward_full_size_sampled():
    """The 0.6B-shaped workload: dq, dr on sampled rows and dk, dv on the last
    keys against the oracle, one by one; the shift invariants over all keys."""
    w = inputs.PREFILL_0P6B
    q, k, v, r = inputs.prefill_inputs_for(w)
    g = torch.Generator().manual_seed(w.seed + 7)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv, dr = _gpu_grads(q, k, v, r, do)
    assert all(torch.isfinite(t).all() for t in (dq, dk, dv, dr))
    rows = sample_rows(w.B, w.Hq, w.L, n_random=6, seed=w.seed)
    rq, rr = ograd.prefill_grad_rows(q, k, v, r, do, rows)
    idx = tuple(torch.as_tensor(x) for x in np.array(rows).T)
    assert_grad_close(dq[idx].numpy(), rq.numpy(), "dq rows")
    assert_grad_close(dr[idx].numpy(), rr.numpy(), "dr rows")
    keys = [(0, 0, w.L - 1), (3, 7, w.L - 2), (1, 4, w.L - 4)]
    rk, rv = ograd.prefill_grad_keys(q, k, v, r, do, keys)
    kidx = tuple(torch.as_tensor(x) for x in np.array(keys).T)
    assert_grad_close(dk[kidx].numpy(), rk.numpy(), "dk last keys")
    assert_grad_close(dv[kidx].numpy(), rv.numpy(), "dv last keys")
    # k-shift invariance: the key gradients of a kv head sum to zero;
    # v-shift equivariance: the value gradients sum to the heads' dout.
    G = w.Hq // w.Hkv
    scale_k = dk.abs().sum(2)
    assert torch.all(dk.sum(2).abs() <= 2e-3 * scale_k + 1e-3)
    want_v = do.double().sum(2).reshape(w.B, w.Hkv, G, w.d).sum(2)
    scale_v = dv.abs().sum(2)
    assert torch.all((dv.sum(2) - want_v).abs() <= 2e-3 * scale_v + 1e-3)


def test_backward_1p7b_shape_sampled():
    """The 1.7B-shaped prefill (B = 1, L = 16384): dq, dr on sampled rows and
    dk, dv on the last keys against the oracle, shift invariants over all keys."""
    w = inputs.PREFILL_1P7B
    q, k, v, r = inputs.prefill_inputs_for(w)
    g = torch.Generator().manual_seed(w.seed + 7)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv, dr = _gpu_grads(q, k, v, r, do)
    rows = sample_rows(w.B, w.Hq, w.L, n_random=4, seed=w.seed)
    rq, rr = ograd.prefill_grad_rows(q, k, v, r, do, rows)
    idx = tuple(torch.as_tensor(x) for x in np.array(rows).T)
    assert_grad_close(dq[idx].numpy(), rq.numpy(), "dq rows (1.7B)")
    assert_grad_close(dr[idx].numpy(), rr.numpy(), "dr rows (1.7B)")
    keys = [(0, 0, w.L - 1), (0, 5, w.L - 3)]
    rk, rv = ograd.prefill_grad_keys(q, k, v, r, do, keys)
    kidx = tuple(torch.as_tensor(x) for x in np.array(keys).T)
    assert_grad_close(dk[kidx].numpy(), rk.numpy(), "dk last keys (1.7B)")
    assert_grad_close(dv[kidx].numpy(), rv.numpy(), "dv last keys (1.7B)")
    G = w.Hq // w.Hkv
    assert torch.all(dk.sum(2).abs() <= 2e-3 * dk.abs().sum(2) + 1e-3)
    want_v = do.double().sum(2).reshape(w.B, w.Hkv, G, w.d).sum(2)
    assert torch.all((dv.sum(2) - want_v).abs() <= 2e-3 * dv.abs().sum(2) + 1e-3)
