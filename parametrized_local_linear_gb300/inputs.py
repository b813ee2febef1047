"""Seeded synthetic inputs for the Parallax forward (no method arithmetic here).

This module only draws random numbers; it is the one piece shared by the
tests, the benchmark and the oracle side. Everything is drawn on the CPU with
a seeded ``torch.Generator`` in fp32 and then cast to the working dtype, so
the same seed gives the same values on any machine. Large tensors are drawn
in chunks so that the fp32 staging never exceeds a few hundred MB.

Value distributions follow the workloads this library is measured on:
q, k, v ~ N(0, 1); the probe r (rho_i = W_R x_i, one per query head) ~
N(0, r_std^2) with r_std = 0.1 for the small fp32 case and 0.05 for the
bf16 model-shaped cases; ragged decode lengths ~ U{lo..hi} inclusive.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

_CHUNK = 1 << 26  # elements drawn per randn call


def _randn(shape, gen, dtype, std=1.0):
    out = torch.empty(shape, dtype=dtype, device=gen.device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = torch.randn(e - s, generator=gen, dtype=torch.float32, device=gen.device)
        if std != 1.0:
            x.mul_(std)
        flat[s:e] = x.to(dtype)
    return out


@dataclass(frozen=True)
class PrefillShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    L: int
    d: int
    dtype: torch.dtype
    r_std: float
    seed: int

    @property
    def pairs(self) -> int:
        """Causal (query, key) pairs j <= i summed over batch and query heads."""
        return self.B * self.Hq * self.L * (self.L + 1) // 2

    @property
    def flops(self) -> int:
        """Algorithmic flops: four length-d dot products per causal pair
        (q.k, r.k, p*v and p*t*v), 2 flops per multiply-add."""
        return 8 * self.d * self.pairs


@dataclass(frozen=True)
class DecodeShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    dtype: torch.dtype
    r_std: float
    seed: int
    len_lo: int
    len_hi: int  # inclusive; equal to len_lo for a uniform batch

    def seqlens(self) -> torch.Tensor:
        gen = torch.Generator().manual_seed(self.seed)
        if self.len_lo == self.len_hi:
            return torch.full((self.B,), self.len_lo, dtype=torch.int32)
        return torch.randint(self.len_lo, self.len_hi + 1, (self.B,), generator=gen,
                             dtype=torch.int64).to(torch.int32)

    def bytes_moved(self, seqlens=None) -> int:
        """Algorithmic HBM bytes: K and V cache read once, q and r read, out
        written (the decode workspace is overhead and not counted)."""
        lens = self.seqlens() if seqlens is None else seqlens
        esz = torch.finfo(self.dtype).bits // 8
        kv = 2 * int(lens.sum()) * self.Hkv * self.d * esz
        return kv + 3 * self.B * self.Hq * self.d * esz


# The five workloads (names say what they are).
TINY_PREFILL_F32 = PrefillShape("tiny_prefill_f32_B1_H2_L256_d64", 1, 2, 2, 256, 64,
                                torch.float32, 0.1, 1001)
PREFILL_0P6B = PrefillShape("prefill_0p6b_B4_Hq16_Hkv8_L4096_d128", 4, 16, 8, 4096, 128,
                            torch.bfloat16, 0.05, 1002)
PREFILL_1P7B = PrefillShape("prefill_1p7b_B1_Hq16_Hkv8_L16384_d128", 1, 16, 8, 16384, 128,
                            torch.bfloat16, 0.05, 1003)
DECODE_B64 = DecodeShape("decode_B64_Hq16_Hkv8_d128_ctx8192", 64, 16, 8, 128,
                         torch.bfloat16, 0.05, 1004, 8192, 8192)
DECODE_RAGGED = DecodeShape("decode_ragged_B8_Hq16_Hkv8_d128_ctx16k_131k", 8, 16, 8, 128,
                            torch.bfloat16, 0.05, 1005, 16384, 131072)
WORKLOADS = {w.name: w for w in (TINY_PREFILL_F32, PREFILL_0P6B, PREFILL_1P7B, DECODE_B64,
                                 DECODE_RAGGED)}


def prefill_inputs(B, Hq, Hkv, L, d, dtype=torch.bfloat16, r_std=0.05, seed=0, device="cpu"):
    """q, k, v, r: q, r [B, Hq, L, d]; k, v [B, Hkv, L, d]. Drawn on the CPU
    unless ``device`` is a CUDA device (then drawn there: same distribution,
    different values; used only where nothing compares against a CPU draw)."""
    gen = torch.Generator(device=device).manual_seed(seed)
    q = _randn((B, Hq, L, d), gen, dtype)
    k = _randn((B, Hkv, L, d), gen, dtype)
    v = _randn((B, Hkv, L, d), gen, dtype)
    r = _randn((B, Hq, L, d), gen, dtype, r_std)
    return q, k, v, r


def prefill_inputs_for(w: PrefillShape, device="cpu"):
    return prefill_inputs(w.B, w.Hq, w.Hkv, w.L, w.d, w.dtype, w.r_std, w.seed, device)


def decode_inputs(B, Hq, Hkv, d, seqlens, dtype=torch.bfloat16, r_std=0.05, seed=0, device="cpu"):
    """q, r [B, Hq, d]; kcache, vcache packed [sum(seqlens), Hkv, d]; seqlens
    int32 [B] (on the CPU). Drawn on ``device`` as in prefill_inputs."""
    seqlens = torch.as_tensor(seqlens, dtype=torch.int32)
    gen = torch.Generator(device=device).manual_seed(seed + 7919)
    T = int(seqlens.sum())
    q = _randn((B, Hq, d), gen, dtype)
    r = _randn((B, Hq, d), gen, dtype, r_std)
    kc = _randn((T, Hkv, d), gen, dtype)
    vc = _randn((T, Hkv, d), gen, dtype)
    return q, r, kc, vc, seqlens


def decode_inputs_for(w: DecodeShape, device="cpu"):
    return decode_inputs(w.B, w.Hq, w.Hkv, w.d, w.seqlens(), w.dtype, w.r_std, w.seed, device)
