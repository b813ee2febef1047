"""Error bound of the FMA-pipe 2^x used for part of the softmax exponentials
(CPU emulation of the device helper's fp32 steps, constants read from the
header so the test checks exactly what the kernel uses)."""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "parametrized_local_linear_gb300", "csrc", "plx_device.cuh")


def _coeffs():
    src = open(HDR).read()
    body = src[src.index("exp2_poly2(uint64_t x)"):]
    body = body[:body.index("return f2(")]
    vals = [v for v in re.findall(r"f2\(([0-9.e-]+)f, \1f\)", body) if not v.startswith("-")]
    # Horner order in the source: c4 (with c3), then c2, c1, c0.
    assert len(vals) == 5, vals
    c4, c3, c2, c1, c0 = (np.float32(v) for v in vals)
    return c0, c1, c2, c3, c4


def _poly_exp2(x):
    c0, c1, c2, c3, c4 = _coeffs()
    shift = np.float32(12582912.0)
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    t = (x + shift).astype(np.float32)
    r = (t - shift).astype(np.float32)
    f = (x - r).astype(np.float32)
    p = c4
    for c in (c3, c2, c1, c0):
        p = (p.astype(np.float64) * f + c).astype(np.float32)  # fused multiply-add, one rounding
    n_bits = (t.view(np.uint32) << np.uint32(23)) - np.uint32((0x4B400000 << 23) & 0xFFFFFFFF)
    return (p.view(np.uint32) + n_bits).view(np.float32)


def test_relative_error_bound():
    x = np.linspace(-125.0, 8.0, 2_000_001).astype(np.float32)
    got = _poly_exp2(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got - ref) / ref) < 4e-6


def test_masked_and_tiny_inputs_clamp_to_negligible():
    x = np.array([-np.inf, -1e30, -500.0, -126.0], dtype=np.float32)
    got = _poly_exp2(x)
    assert np.all(np.isfinite(got)) and np.all(got >= 0) and np.all(got < 2.0 ** -124)


def test_exact_at_zero_and_integers():
    got = _poly_exp2(np.array([0.0, 1.0, -1.0, -20.0, 8.0], dtype=np.float32)).astype(np.float64)
    ref = np.exp2([0.0, 1.0, -1.0, -20.0, 8.0])
    assert np.max(np.abs(got - ref) / ref) < 1e-6
