"""Shared helpers for the parity tests (tolerances, row sampling, device setup)."""
import math
import random

import numpy as np
import torch

# bf16 inputs, fp32 accumulation: max|err| <= 1e-2 * max|o_ref| + 2e-3.
BF16_REL, BF16_ABS = 1e-2, 2e-3
# fp32 path: max|err| / max|o_ref| <= 1e-5 (and the same for lse on |lse|).
F32_REL = 1e-5
# lse of the bf16 prefill, absolute (natural-log units). The kernel forms
# lse = (m + log2 l) ln 2 from fp32 scores and an fp32 sum l of MUFU
# exponentials; bf16 rounding never enters it. Worst-case sources, d = 128,
# up to 16384 keys: the fp32 accumulation of a score from 128 exact bf16
# products, d 2^-24 sum|q_i k_i| tau <= 6e-5 for inputs ~ N(0, 1); the fp32
# sum of l, 64 terms per key tile added to at most 256 tile sums in
# sequence, relative (64 + 256) 2^-24 = 1.9e-5; ex2.approx (2^-22 relative)
# and log2f (2 ulp), below 1e-6. Total under 8e-5; the bound allows 2.5x.
LSE_ABS = 2e-4
# sbar = sigma / l of the training forward, absolute: sigma sums p t in fp32
# with t = rho . k from the same fp32 accumulation (|t| <= 3 at r ~ N(0,
# 0.05^2)), so the summation bound above, 1.9e-5 relative of max|t|, plus the
# accumulation error of t, d 2^-24 sum|r_i k_i| <= 3e-5, stays below 1e-4;
# the bound allows 2x.
SBAR_ABS = 2e-4


def device():
    from parametrized_local_linear_gb300 import build
    build.build()
    return torch.device("cuda", 0)


def assert_bf16_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.max(np.abs(got - ref)) if got.size else 0.0
    bound = BF16_REL * np.max(np.abs(ref)) + BF16_ABS if ref.size else 0.0
    assert err <= bound, f"{what}: max|err| {err:.3e} > {bound:.3e}"
    return err, bound


def assert_f32_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel = np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30)
    assert rel <= F32_REL, f"{what}: relative error {rel:.3e} > {F32_REL:.0e}"
    return rel


def sample_rows(B, Hq, L, n_random, seed):
    """The fixed edge rows of every tile boundary that matters plus a seeded
    random set, spread over (batch, head)."""
    rng = random.Random(seed)
    fixed = sorted({i for i in (0, 1, 63, 64, 127, 128, 129, L // 2, L - 2, L - 1) if 0 <= i < L})
    rows = set()
    for n, i in enumerate(fixed):
        rows.add((n % B, (3 * n) % Hq, i))
    rows.add((B - 1, Hq - 1, L - 1))
    while len(rows) < len(fixed) + 1 + n_random:
        rows.add((rng.randrange(B), rng.randrange(Hq), rng.randrange(L)))
    return sorted(rows)


def tolerance_note():
    return f"bf16: {BF16_REL}*max|ref| + {BF16_ABS}; fp32: {F32_REL} relative"


def tau(d):
    return 1.0 / math.sqrt(d)


# Correction-to-output ratio cor = |Sigma rho| / |o| from the bf16 kernels:
# a bound per row, derived from the roundings that reach the two norms. The
# kernels round every weight p_j and product p_j t_j (t_j = rho . k_j) to
# bf16 before the value products (relative error at most 2^-8 each: bf16
# keeps 8 significant bits, rounded to nearest) and form
# both norms from the fp32 correction O2 - O1 s and output O1 - (O2 - O1 s)
# before o is rounded. With w the normalised weights, s = sum w t,
# A = sum_j w_j |v_j| and C = sum_j w_j |t_j| |v_j| (Euclidean norms), the
# correction moves by at most E_c = 2^-8 (C + |s| A) and o by at most
# E_o = 2^-8 (1 + |s|) A + E_c, so the ratio moves by at most
# (E_c + cor E_o) / (|o| - E_o). A row that sees one key has Sigma = 0, yet
# the kernel's ratio there is |bf16(t) - t| <= 2^-8 |t|: the bound
# covers it through C. The fp32 accumulations (relative 2e-5 at most here)
# are covered by raising 2^-8 by 2%.
_COR_EPS = 2.0 ** -8 * 1.02


def _cor_bound_rows(Q, R, K, V, nkeys):
    """Bounds for query rows Q, R (torch fp64 [n, d]) over keys K, V, row i
    seeing keys 0 .. nkeys[i] - 1."""
    n, d = Q.shape
    nk = int(nkeys.max())
    K, V = K[:nk], V[:nk]
    S = (Q @ K.T) / math.sqrt(d)
    S = S.masked_fill(torch.arange(nk)[None, :] >= nkeys[:, None], -math.inf)
    w = torch.softmax(S, dim=1)
    t = R @ K.T
    s = (w * t).sum(1)
    vn = V.norm(dim=1)
    A = w @ vn
    C = (w * t.abs()) @ vn
    O1 = w @ V
    corr = (w * t) @ V - O1 * s[:, None]
    on = (O1 - corr).norm(dim=1)
    cor = corr.norm(dim=1) / on
    Ec = _COR_EPS * (C + s.abs() * A)
    Eo = _COR_EPS * (1 + s.abs()) * A + Ec
    room = on - Eo
    return torch.where(room > 0, (Ec + cor * Eo) / room.clamp_min(1e-300),
                       torch.full_like(on, math.inf)).numpy()


def cor_bounds_prefill(q, k, v, r, rows=None, row_block=512):
    """Per-row COR bounds of a (chunked) causal prefill: [B, Hq, Lq] for
    rows=None, else [n] for the listed (b, h, i)."""
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    G, off = Hq // Hkv, Lk - Lq
    f = lambda x: x.detach().to("cpu", torch.float64)  # noqa: E731
    if rows is not None:
        out = np.empty(len(rows))
        for n, (b, h, i) in enumerate(rows):
            out[n] = _cor_bound_rows(f(q[b, h, i:i + 1]), f(r[b, h, i:i + 1]), f(k[b, h // G]),
                                     f(v[b, h // G]), torch.tensor([off + i + 1]))[0]
        return out
    out = np.empty((B, Hq, Lq))
    for b in range(B):
        for h in range(Hq):
            K, V, Q, R = f(k[b, h // G]), f(v[b, h // G]), f(q[b, h]), f(r[b, h])
            for i0 in range(0, Lq, row_block):
                i1 = min(Lq, i0 + row_block)
                out[b, h, i0:i1] = _cor_bound_rows(Q[i0:i1], R[i0:i1], K, V,
                                                   off + torch.arange(i0, i1) + 1)
    return out


def cor_bounds_decode(q, r, kc, vc, seqlens):
    """Per-(sequence, head) COR bounds of a decode: [B, Hq]; 0 for an empty
    sequence (its ratio is 0 by definition on both sides)."""
    B, Hq, d = q.shape
    G = Hq // kc.shape[1]
    lens = [int(x) for x in seqlens.tolist()]
    offs = np.concatenate([[0], np.cumsum(lens)])
    f = lambda x: x.detach().to("cpu", torch.float64)  # noqa: E731
    out = np.zeros((B, Hq))
    for b in range(B):
        if lens[b] == 0:
            continue
        for h in range(Hq):
            out[b, h] = _cor_bound_rows(f(q[b, h:h + 1]), f(r[b, h:h + 1]),
                                        f(kc[offs[b]:offs[b + 1], h // G]),
                                        f(vc[offs[b]:offs[b + 1], h // G]),
                                        torch.tensor([lens[b]]))[0]
    return out


def assert_cor_close(got, ref, bound, what=""):
    """|cor_gpu - cor_ref| <= bound per row (bounds from cor_bounds_*)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape == np.shape(bound), (got.shape, ref.shape, np.shape(bound))
    assert np.all(np.isfinite(got)) and np.all(got >= 0), f"{what}: bad ratio"
    excess = np.abs(got - ref) / np.maximum(bound, 1e-300)
    worst = int(np.argmax(excess)) if got.size else 0
    if got.size:
        print(f"{what}: max |cor err| / bound = {excess.flat[worst]:.3f}")
    assert not got.size or excess.flat[worst] <= 1.0, (
        f"{what}: cor {got.flat[worst]:.5f} vs {ref.flat[worst]:.5f}, bound "
        f"{np.ravel(bound)[worst]:.2e}")
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


# Gradients from the bf16 backward: the kernels round w c, tau ds and dt to
# bf16 before the gradient GEMMs (2^-8 relative per term), read o and o^SA as
# bf16, and round the result to bf16 (2^-8 again). The term roundings are
# independent across the keys (or queries) a gradient sums, so they largely
# cancel; the output rounding alone reaches 2^-8 = 0.39% of an element. The
# bound, 1e-2 of the tensor's largest gradient, is the output tolerance of
# the forward applied per gradient tensor: 2.5x the output rounding of the
# largest element. Measured: at most 0.67% on every tested shape.
GRAD_REL = 1e-2


def assert_grad_close(got, ref, what="", scale=None):
    """max|err| <= GRAD_REL * scale, scale = max|ref| unless given."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite gradient"
    err = np.max(np.abs(got - ref))
    scale = np.max(np.abs(ref)) if scale is None else scale
    print(f"{what}: max|err| / max|ref| = {err / scale:.3e}")
    assert err <= GRAD_REL * scale, f"{what}: max|err| {err:.3e} > {GRAD_REL} * {scale:.3e}"
    return err / scale
