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


# Correction-to-output ratio |Sigma rho| / |o| from the bf16 kernels: both
# norms come from fp32 accumulators fed by bf16-rounded P and P*T (relative
# rounding 2^-9 per weight), so the relative factor of the output tolerance
# (5x that rounding, headroom for the cancellation in O2 - O1*s) carries over;
# the absolute floor covers rows whose ratio is near 0.
COR_REL, COR_ABS = 1e-2, 2e-3


def assert_cor_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)) and np.all(got >= 0), f"{what}: bad ratio"
    excess = np.abs(got - ref) - (COR_REL * ref + COR_ABS)
    worst = int(np.argmax(excess)) if got.size else 0
    assert not got.size or excess.flat[worst] <= 0, (
        f"{what}: cor {got.flat[worst]:.5f} vs {ref.flat[worst]:.5f}")
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


# Gradients from the bf16 backward: the kernels round w c, tau ds and dt to
# bf16 before the gradient GEMMs (2^-9 relative per term), read o and o^SA as
# bf16, and round the result to bf16; the relative factor allows 5x those
# roundings against the largest gradient of the tensor.
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
