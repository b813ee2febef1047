"""Pins for the fp64 oracle against things other than itself (CPU only).

Each test targets a mistake the oracle could plausibly contain: a dropped
centring term, a wrong sign, a transposed Sigma, a wrong GQA head mapping, an
off-by-one in the causal window, or a bad softmax normaliser.

Definition pinned (page "Parallax: parametrized local linear attention for
language modeling", section "Core mechanism", output equation):
o_i = o^SA_i - Sigma_KV^(i) rho_i, with Sigma_KV^(i) the softmax-weighted,
centred KV cross-covariance of the keys query i sees.
"""
import glob
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import expanded
from parametrized_local_linear_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_fixture(path):
    rec = {"k": [], "v": []}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            vals = [float(x) for x in vals]
            if key in ("k", "v"):
                rec[key].append(vals)
            else:
                rec[key] = vals
    return rec


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN, "hand_*.txt"))))
def test_hand_worked_examples(path):
    rec = _parse_fixture(path)
    d = len(rec["q"])
    o, lse, sig = oracle.query(np.array(rec["q"]), np.array(rec["rho"]), np.array(rec["k"]),
                               np.array(rec["v"]), tau=rec["tau"][0], with_sigma=True)
    np.testing.assert_allclose(o, rec["out"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rec["lse"][0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sig.reshape(-1), rec["sigma"], rtol=0, atol=1e-12)
    assert sig.shape == (d, d)


def _small(B=2, Hq=4, Hkv=2, L=24, d=8, seed=3, r_std=0.3):
    return inputs.prefill_inputs(B, Hq, Hkv, L, d, torch.float64, r_std, seed)


def test_row0_closed_form():
    """Row 0 sees one key: weight 1, Sigma = 0, so o = v_0 whatever rho is."""
    q, k, v, r = _small()
    out, lse = oracle.prefill(q, k, v, r)
    G = q.shape[1] // k.shape[1]
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            np.testing.assert_allclose(out[b, h, 0], v[b, h // G, 0].numpy(), rtol=0, atol=1e-14)
            s0 = float(q[b, h, 0] @ k[b, h // G, 0]) / math.sqrt(q.shape[-1])
            assert abs(lse[b, h, 0] - s0) < 1e-12


def test_row1_closed_form():
    """Row 1 sees two keys: Sigma = w0 w1 (v1 - v0)(k1 - k0)^T."""
    q, k, v, r = _small(seed=11)
    out, _ = oracle.prefill(q, k, v, r)
    d = q.shape[-1]
    G = q.shape[1] // k.shape[1]
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            K = k[b, h // G, :2].numpy(); V = v[b, h // G, :2].numpy()
            qi = q[b, h, 1].numpy(); ri = r[b, h, 1].numpy()
            s = K @ qi / math.sqrt(d)
            w1 = 1.0 / (1.0 + math.exp(s[0] - s[1])); w0 = 1.0 - w1
            osa = w0 * V[0] + w1 * V[1]
            want = osa - w0 * w1 * (V[1] - V[0]) * float((K[1] - K[0]) @ ri)
            np.testing.assert_allclose(out[b, h, 1], want, rtol=0, atol=1e-12)


def test_rho_zero_is_softmax_attention():
    """W_R = 0 (rho = 0) reduces Parallax to causal softmax attention: pinned to
    torch's fp64 scaled_dot_product_attention with KV heads repeated for GQA."""
    q, k, v, r = _small(B=2, Hq=6, Hkv=2, L=40, d=16, seed=5)
    out, lse = oracle.prefill(q, k, v, torch.zeros_like(r))
    G = q.shape[1] // k.shape[1]
    kk = k.repeat_interleave(G, dim=1); vv = v.repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=True)
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)
    L = q.shape[2]
    scores = (q @ kk.transpose(-1, -2)) / math.sqrt(q.shape[-1])
    mask = torch.ones(L, L, dtype=torch.bool).tril()
    ref_lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("n,d", [(1, 3), (5, 4), (37, 8), (200, 16)])
def test_sigma_is_weighted_covariance(n, d):
    """Sigma equals the V-K block of numpy's weighted (biased) covariance with
    the softmax weights as analytic weights; softmax from scipy."""
    rng = np.random.default_rng(n * 100 + d)
    q = rng.normal(size=d); rho = rng.normal(size=d)
    K = rng.normal(size=(n, d)); V = rng.normal(size=(n, d))
    o, lse, sig = oracle.query(q, rho, K, V, with_sigma=True)
    w = scipy.special.softmax(K @ q / math.sqrt(d))
    if n == 1:
        ref = np.zeros((d, d))
    else:
        ref = np.cov(np.vstack([V.T, K.T]), aweights=w, bias=True)[:d, d:]
    np.testing.assert_allclose(sig, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, w @ V - ref @ rho, rtol=0, atol=1e-12)
    assert abs(lse - scipy.special.logsumexp(K @ q / math.sqrt(d))) < 1e-12


def test_uniform_weights_give_population_covariance():
    rng = np.random.default_rng(7)
    n, d = 9, 5
    K = rng.normal(size=(n, d)); V = rng.normal(size=(n, d)); rho = rng.normal(size=d)
    _, _, sig = oracle.query(np.zeros(d), rho, K, V, with_sigma=True)
    ref = np.cov(V.T, K.T, bias=True)[:d, d:]
    np.testing.assert_allclose(sig, ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("d,L,Lk,Hq,Hkv,block", [
    (4, 16, 16, 2, 2, 16), (8, 33, 33, 4, 2, 7), (64, 64, 64, 4, 1, 64), (8, 20, 45, 4, 2, 6)])
def test_expanded_form_matches_the_explicit_oracle(d, L, Lk, Hq, Hkv, block):
    """The expanded fp64 form O1 - O2 + O1*s (dense matrices, query rows in
    blocks) against the explicit-Sigma oracle: every row, lse too, with a
    chunk offset in the last case. A dropped term, a wrong sign, an unscaled
    score or a wrong causal window in either would show here."""
    q, k, v, r = _small(B=2, Hq=Hq, Hkv=Hkv, L=Lk, d=d, seed=d + L)
    q, r = q[:, :, Lk - L:], r[:, :, Lk - L:]
    out, lse, cor = oracle.prefill(q, k, v, r, with_cor=True)
    eo, e_lse, _, _, ecor = expanded.prefill(q, k, v, r, row_block=block, with_parts=True)
    np.testing.assert_allclose(eo, out, rtol=0, atol=1e-11)
    np.testing.assert_allclose(e_lse, lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ecor, cor, rtol=1e-10, atol=1e-12)


def test_expanded_parts_against_library_routines():
    """o^SA of the expanded form is torch's causal SDPA (fp64, GQA by repeat);
    sbar is rho . mu with mu the softmax-weighted key mean from numpy."""
    q, k, v, r = _small(B=1, Hq=4, Hkv=2, L=19, d=8, seed=71)
    _, _, osa, sbar, _ = expanded.prefill(q, k, v, r, row_block=5, with_parts=True)
    kk, vv = k.repeat_interleave(2, dim=1), v.repeat_interleave(2, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=True)
    np.testing.assert_allclose(osa, ref.numpy(), rtol=0, atol=1e-12)
    for h, i in ((0, 0), (1, 7), (3, 18)):
        w = scipy.special.softmax(kk[0, h, :i + 1].numpy() @ q[0, h, i].numpy() / math.sqrt(8))
        mu = np.average(kk[0, h, :i + 1].numpy(), axis=0, weights=w)
        assert abs(sbar[0, h, i] - r[0, h, i].numpy() @ mu) < 1e-12


def test_expanded_decode_matches_the_explicit_oracle():
    lens = [5, 0, 17, 1, 40]
    q, r, kc, vc, sl = inputs.decode_inputs(len(lens), 4, 2, 8, lens, torch.float64, 0.3, 9)
    out, lse, cor = oracle.decode(q, r, kc, vc, sl, with_cor=True)
    eo, e_lse, ecor = expanded.decode(q, r, kc, vc, sl, with_cor=True)
    np.testing.assert_allclose(eo, out, rtol=0, atol=1e-11)
    np.testing.assert_allclose(ecor, cor, rtol=1e-10, atol=1e-12)
    live = np.array(lens) > 0
    np.testing.assert_allclose(e_lse[live], lse[live], rtol=0, atol=1e-12)
    assert np.all(eo[1] == 0) and np.all(ecor[1] == 0)


def test_shift_v_shifts_output():
    q, k, v, r = _small(seed=21)
    c = torch.linspace(-2, 3, q.shape[-1], dtype=torch.float64)
    o0, _ = oracle.prefill(q, k, v, r)
    o1, _ = oracle.prefill(q, k, v + c, r)
    np.testing.assert_allclose(o1, o0 + c.numpy(), rtol=0, atol=1e-11)


def test_shift_k_leaves_output_unchanged():
    """A common shift of every key changes each score by q.c (the same for every
    key of a row), so the weights, o^SA and the centred Sigma do not move."""
    q, k, v, r = _small(seed=22)
    c = torch.linspace(1, -1, q.shape[-1], dtype=torch.float64)
    o0, _ = oracle.prefill(q, k, v, r)
    o1, _ = oracle.prefill(q, k + c, v, r)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-11)


def test_uncentred_covariance_would_fail_the_k_shift_pin():
    """The k-shift pin discriminates: an uncentred sum_j w_j v_j k_j^T does move."""
    rng = np.random.default_rng(4)
    n, d = 12, 6
    q = rng.normal(size=d); rho = rng.normal(size=d)
    K = rng.normal(size=(n, d)); V = rng.normal(size=(n, d)); c = np.full(d, 0.7)

    def uncentred(K):
        w = scipy.special.softmax(K @ q / math.sqrt(d))
        return w @ V - (V.T * w) @ K @ rho

    assert np.max(np.abs(uncentred(K + c) - uncentred(K))) > 1e-3
    o0, _ = oracle.query(q, rho, K, V)
    o1, _ = oracle.query(q, rho, K + c, V)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)


def test_correction_is_linear_in_rho():
    q, k, v, r = _small(seed=23)
    r2 = _small(seed=24)[3]
    base, _ = oracle.prefill(q, k, v, torch.zeros_like(r))
    oa, _ = oracle.prefill(q, k, v, r)
    ob, _ = oracle.prefill(q, k, v, r2)
    oab, _ = oracle.prefill(q, k, v, 2.5 * r - 0.5 * r2)
    np.testing.assert_allclose(oab - base, 2.5 * (oa - base) - 0.5 * (ob - base), rtol=0, atol=1e-11)


def test_equal_keys_remove_the_correction():
    """All keys equal: k_j - mu = 0, Sigma = 0, o = o^SA (uniform average of v)."""
    q, k, v, r = _small(seed=25)
    k = k[:, :, :1].expand_as(k).contiguous()
    out, _ = oracle.prefill(q, k, v, r)
    G = q.shape[1] // k.shape[1]
    L = q.shape[2]
    cum = torch.cumsum(v, dim=2) / torch.arange(1, L + 1, dtype=torch.float64)[:, None]
    np.testing.assert_allclose(out, cum.repeat_interleave(G, dim=1).numpy(), rtol=0, atol=1e-12)


def test_decode_equals_last_prefill_row():
    """A decode query over a packed ragged cache equals the last causal row of a
    prefill over the same keys (checks the packed-offset walk)."""
    Hq, Hkv, d = 4, 2, 8
    lens = [5, 1, 17, 9]
    q, r, kc, vc, sl = inputs.decode_inputs(len(lens), Hq, Hkv, d, lens, torch.float64, 0.3, 9)
    out, lse = oracle.decode(q, r, kc, vc, sl)
    off = 0
    for b, n in enumerate(lens):
        kb = kc[off:off + n].permute(1, 0, 2)[None]
        vb = vc[off:off + n].permute(1, 0, 2)[None]
        qb = torch.zeros(1, Hq, n, d, dtype=torch.float64); rb = torch.zeros_like(qb)
        qb[0, :, -1] = q[b]; rb[0, :, -1] = r[b]
        po, pl = oracle.prefill(qb, kb, vb, rb, rows=[(0, h, n - 1) for h in range(Hq)])
        np.testing.assert_allclose(out[b], po, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], pl, rtol=0, atol=1e-13)
        off += n


def test_decode_empty_sequence_is_zero():
    q, r, kc, vc, sl = inputs.decode_inputs(3, 2, 1, 4, [3, 0, 2], torch.float64, 0.3, 1)
    out, lse = oracle.decode(q, r, kc, vc, sl)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(out[[0, 2]]))


def test_row_sampling_matches_full_pass():
    q, k, v, r = _small(B=1, Hq=2, Hkv=1, L=30, d=8, seed=31)
    full, flse = oracle.prefill(q, k, v, r)
    rows = [(0, 1, 29), (0, 0, 0), (0, 1, 7)]
    o, l = oracle.prefill(q, k, v, r, rows=rows)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(o[n], full[b, h, i]) and l[n] == flse[b, h, i]


def test_chunked_prefill_is_the_tail_of_the_full_prefill():
    """A chunk of Lq queries over Lk keys (query i sees keys 0..Lk-Lq+i) is the
    last Lq rows of the full causal prefill over the same keys."""
    q, k, v, r = _small(B=1, Hq=4, Hkv=2, L=40, d=8, seed=41)
    full, flse = oracle.prefill(q, k, v, r)
    for lq in (1, 7, 40):
        out, lse = oracle.prefill(q[:, :, -lq:].contiguous(), k, v, r[:, :, -lq:].contiguous())
        np.testing.assert_array_equal(out, full[:, :, -lq:])
        np.testing.assert_array_equal(lse, flse[:, :, -lq:])


# --- COR: the correction-to-output ratio |Sigma rho| / |o| per query ---------
# (the page's experimental results report COR per layer; the pages give no
# formula, and the ratio of Euclidean norms per query is the reading pinned.)

@pytest.mark.parametrize("n,d", [(2, 3), (17, 8), (150, 16)])
def test_cor_against_library_covariance(n, d):
    """COR from numpy's weighted covariance and scipy's softmax, with o built
    from those too: catches a ratio taken against o^SA instead of o, a squared
    norm, or the wrong branch in the numerator."""
    rng = np.random.default_rng(n * 31 + d)
    q = rng.normal(size=d); rho = rng.normal(size=d) * 0.3
    K = rng.normal(size=(n, d)); V = rng.normal(size=(n, d))
    _, _, cor = oracle.query(q, rho, K, V, with_cor=True)
    w = scipy.special.softmax(K @ q / math.sqrt(d))
    sig = np.cov(np.vstack([V.T, K.T]), aweights=w, bias=True)[:d, d:]
    corr = sig @ rho
    ref = np.linalg.norm(corr) / np.linalg.norm(w @ V - corr)
    assert abs(cor - ref) <= 1e-12 * max(1.0, ref)


def test_cor_two_keys_closed_form():
    """Two keys: |Sigma rho| = w0 w1 |(k1 - k0).rho| |v1 - v0|."""
    rng = np.random.default_rng(12)
    d = 6
    q = rng.normal(size=d); rho = rng.normal(size=d)
    K = rng.normal(size=(2, d)); V = rng.normal(size=(2, d))
    o, _, cor = oracle.query(q, rho, K, V, with_cor=True)
    s = K @ q / math.sqrt(d)
    w0 = 1.0 / (1.0 + math.exp(s[1] - s[0])); w1 = 1.0 - w0
    num = w0 * w1 * abs((K[1] - K[0]) @ rho) * math.sqrt(((V[1] - V[0]) ** 2).sum())
    assert abs(cor - num / math.sqrt((o ** 2).sum())) < 1e-12


def test_cor_zero_cases():
    """One key (Sigma = 0), rho = 0, and an empty key set all give 0."""
    rng = np.random.default_rng(13)
    d = 5
    q = rng.normal(size=d); rho = rng.normal(size=d)
    K = rng.normal(size=(7, d)); V = rng.normal(size=(7, d))
    assert oracle.query(q, rho, K[:1], V[:1], with_cor=True)[2] == 0.0
    assert oracle.query(q, np.zeros(d), K, V, with_cor=True)[2] == 0.0
    assert oracle.query(q, rho, K[:0], V[:0], with_cor=True)[2] == 0.0


def test_cor_is_invariant_to_value_scale():
    """Scaling every v by c > 0 scales both Sigma rho and o by c."""
    rng = np.random.default_rng(14)
    d = 8
    q = rng.normal(size=d); rho = rng.normal(size=d)
    K = rng.normal(size=(30, d)); V = rng.normal(size=(30, d))
    c1 = oracle.query(q, rho, K, V, with_cor=True)[2]
    c2 = oracle.query(q, rho, K, 3.5 * V, with_cor=True)[2]
    assert c1 > 0 and abs(c1 - c2) < 1e-12 * c1


def test_cor_prefill_and_decode_agree_with_query():
    """The batched walks return the per-query ratio (GQA mapping, causal
    window and packing as for the outputs)."""
    g = torch.Generator().manual_seed(15)
    B, Hq, Hkv, L, d = 2, 4, 2, 9, 8
    q, k, v, r = (torch.randn(B, h, L, d, generator=g, dtype=torch.float64) for h in (Hq, Hkv, Hkv, Hq))
    _, _, cor = oracle.prefill(q, k, v, r, with_cor=True)
    for b, h, i in [(0, 0, 0), (0, 3, 4), (1, 2, 8), (1, 1, 1)]:
        ref = oracle.query(q[b, h, i].numpy(), r[b, h, i].numpy(), k[b, h // 2, :i + 1].numpy(),
                           v[b, h // 2, :i + 1].numpy(), with_cor=True)[2]
        assert abs(cor[b, h, i] - ref) < 1e-14
    seqlens = torch.tensor([9, 0])
    kc = torch.cat([k[0].transpose(0, 1), k[1, :, :0].transpose(0, 1)])
    vc = torch.cat([v[0].transpose(0, 1), v[1, :, :0].transpose(0, 1)])
    _, _, dcor = oracle.decode(q[:, :, -1], r[:, :, -1], kc, vc, seqlens, with_cor=True)
    np.testing.assert_allclose(dcor[0], cor[0, :, -1], rtol=0, atol=1e-14)
    assert np.all(dcor[1] == 0.0)


# --- the fused probe projection [W_Q; W_K; W_V; W_R] x -----------------------

def test_projection_matches_brute_force_loops():
    rng = np.random.default_rng(21)
    B, L, D, Hq, Hkv, d = 2, 3, 5, 2, 1, 2
    F = (2 * Hq + 2 * Hkv) * d
    x = rng.normal(size=(B * L, D)); w = rng.normal(size=(F, D))
    q, k, v, r = oracle.qkvr_projection(x, w, B, L, Hq, Hkv, d)
    parts = [(q, 0, Hq), (k, Hq * d, Hkv), (v, (Hq + Hkv) * d, Hkv), (r, (Hq + 2 * Hkv) * d, Hq)]
    for out, base, H in parts:
        assert out.shape == (B, H, L, d)
        for b in range(B):
            for h in range(H):
                for l in range(L):
                    for e in range(d):
                        f = base + h * d + e
                        ref = sum(x[b * L + l, c] * w[f, c] for c in range(D))
                        assert abs(out[b, h, l, e] - ref) < 1e-12


def test_projection_head_layout_with_selector_weights():
    """Unit-vector rows make each output element a copy of one input element,
    so a transposed head or token index shows up exactly."""
    B, L, Hq, Hkv, d = 2, 4, 2, 1, 3
    F = (2 * Hq + 2 * Hkv) * d
    D = F
    x = np.arange(B * L * D, dtype=np.float64).reshape(B * L, D)
    w = np.eye(F)
    q, k, v, r = oracle.qkvr_projection(x, w, B, L, Hq, Hkv, d)
    assert q[1, 1, 2, 0] == x[1 * L + 2, 1 * d + 0]
    assert k[0, 0, 3, 2] == x[3, Hq * d + 2]
    assert v[1, 0, 0, 1] == x[L, (Hq + Hkv) * d + 1]
    assert r[0, 1, 1, 2] == x[1, (Hq + 2 * Hkv) * d + d + 2]


def test_zero_probe_weights_give_softmax_attention():
    """W_R = 0 (the pages' start for adapting a pretrained model) makes rho
    zero, and the layer output is then softmax attention."""
    rng = np.random.default_rng(22)
    B, L, D, Hq, Hkv, d = 1, 9, 8, 2, 1, 4
    F = (2 * Hq + 2 * Hkv) * d
    x = rng.normal(size=(B * L, D)); w = rng.normal(size=(F, D))
    w[(Hq + 2 * Hkv) * d:] = 0.0
    q, k, v, r = oracle.qkvr_projection(x, w, B, L, Hq, Hkv, d)
    assert np.all(r == 0.0)
    out, _ = oracle.prefill(q, k, v, r)
    t = [torch.from_numpy(a) for a in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(
        t[0], t[1].repeat_interleave(2, dim=1), t[2].repeat_interleave(2, dim=1), is_causal=True)
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)
