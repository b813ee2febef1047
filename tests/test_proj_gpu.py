"""GPU fused input projection [W_Q; W_K; W_V; W_R] x against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from parametrized_local_linear_gb300 import (plx_check_device_error, plx_prefill_fwd,
                                             plx_qkvr_proj)

from helpers import assert_bf16_close, device

pytestmark = pytest.mark.gpu

# The kernel rounds an fp32 sum once to bf16 (nearest even): at most half a
# bf16 unit in the last place, 2^-8 relative; fp32 accumulation over D terms
# adds far less than the small absolute allowance.
ROUND_REL = 2.0 ** -8


def _weights(F, D, seed, zero_probe_from=None):
    g = torch.Generator().manual_seed(seed)
    x_std = 1.0
    w = torch.randn(F, D, generator=g) / D ** 0.5
    if zero_probe_from is not None:
        w[zero_probe_from:] = 0.0
    return w.to(torch.bfloat16), x_std


def _inputs(B, L, D, Hq, Hkv, seed, zero_probe=False):
    F = (2 * Hq + 2 * Hkv) * 128
    w, _ = _weights(F, D, seed, (Hq + 2 * Hkv) * 128 if zero_probe else None)
    g = torch.Generator().manual_seed(seed + 1)
    x = torch.randn(B * L, D, generator=g).to(torch.bfloat16)
    return x, w


def _check_rounding(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bound = ROUND_REL * np.abs(ref) + 1e-6 * np.max(np.abs(ref))
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"{what}: {got[worst]} vs {ref[worst]} at {worst}"


@pytest.mark.parametrize("B,L,D,Hq,Hkv", [
    (1, 1, 64, 1, 1),        # a single token
    (1, 128, 64, 1, 1),      # one tile of each kind
    (3, 129, 2048, 1, 1),    # an odd number of token tiles (the cluster's last partner is empty)
    (2, 200, 1024, 2, 1),    # a 128-row tile straddles the two sequences
    (1, 77, 200, 3, 1),      # token tail and a K tail (200 = 3 x 64 + 8)
    (3, 50, 512, 4, 2),      # several sequences inside one tile
])
def test_projection_matches_oracle(B, L, D, Hq, Hkv):
    dev = device()
    x, w = _inputs(B, L, D, Hq, Hkv, 100 + L)
    outs = plx_qkvr_proj(x.to(dev), w.to(dev), B, L, Hq, Hkv)
    plx_check_device_error()
    refs = oracle.qkvr_projection(x, w, B, L, Hq, Hkv, 128)
    for name, got, ref in zip("qkvr", outs, refs):
        _check_rounding(got.double().cpu().numpy(), ref, name)


@pytest.mark.parametrize("D", [1024, 2048])
def test_projection_full_size_sampled_tokens(D):
    """The 0.6B- and 1.7B-shaped layers (model dims 1024 and 2048, 16 query
    and 8 kv heads, B = 4, L = 4096 tokens) on sampled token rows."""
    B, L, Hq, Hkv = 4, 4096, 16, 8
    dev = device()
    x, w = _inputs(B, L, D, Hq, Hkv, 7)
    q, k, v, r = plx_qkvr_proj(x.to(dev), w.to(dev), B, L, Hq, Hkv)
    plx_check_device_error()
    rng = np.random.default_rng(3)
    toks = np.unique(np.concatenate([[0, 127, 128, L - 1, L, B * L - 1], rng.integers(0, B * L, 40)]))
    y = x[toks].double().numpy() @ w.double().numpy().T  # [n, F]
    F_q, F_k = Hq * 128, Hkv * 128
    for n, t in enumerate(toks):
        b, l = divmod(int(t), L)
        got = torch.cat([q[b, :, l].reshape(-1), k[b, :, l].reshape(-1), v[b, :, l].reshape(-1),
                         r[b, :, l].reshape(-1)]).double().cpu().numpy()
        assert got.shape[0] == 2 * F_q + 2 * F_k
        _check_rounding(got, y[n], f"token {t}")


def test_zero_probe_weights_give_zero_rho_and_softmax_attention():
    dev = device()
    B, L, D, Hq, Hkv = 1, 300, 256, 2, 1
    x, w = _inputs(B, L, D, Hq, Hkv, 9, zero_probe=True)
    q, k, v, r = plx_qkvr_proj(x.to(dev), w.to(dev), B, L, Hq, Hkv)
    assert torch.all(r == 0)
    out, _ = plx_prefill_fwd(q, k, v, r)
    plx_check_device_error()
    ref, _ = oracle.prefill(q.cpu(), k.cpu(), v.cpu(), r.cpu())
    assert_bf16_close(out.double().cpu().numpy(), ref, "W_R = 0 layer")


def test_projection_writes_nothing_outside_its_outputs():
    dev = device()
    B, L, D, Hq, Hkv = 2, 70, 128, 1, 1
    x, w = _inputs(B, L, D, Hq, Hkv, 11)
    n = B * Hq * L * 128
    buf = torch.full((4 * n + 4 * 4096,), float("nan"), dtype=torch.bfloat16, device=dev)
    views = []
    for i in range(4):
        off = 2048 + i * (n + 4096)
        views.append(buf[off:off + n].view(B, Hq, L, 128))
    plx_qkvr_proj(x.to(dev), w.to(dev), B, L, Hq, Hkv, q=views[0], k=views[1], v=views[2],
                  r=views[3])
    plx_check_device_error()
    mask = torch.ones_like(buf, dtype=torch.bool)
    for i in range(4):
        off = 2048 + i * (n + 4096)
        mask[off:off + n] = False
    assert torch.isnan(buf[mask]).all()
    assert not torch.isnan(buf[~mask]).any()
