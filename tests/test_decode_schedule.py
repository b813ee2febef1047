"""The decode's share schedule, restated in Python and checked on random
batches: every key of every (sequence, kv head) row belongs to exactly one
share; the record slot c + row of each (share, row) pair that meets is
distinct and inside the workspace; the row table {first slot, slots} names
exactly the shares that hold the row; the position-to-share formula inverts
the share boundaries; and the default share count keeps its stated bounds.
The CUDA split kernel computes the same integer formulas on the device (its
parity against the oracle is in test_decode_gpu.py); this test pins the
formulas themselves.
"""
import math
import random

import pytest


def share_count(lens, Hkv, nshare, default):
    """Explicit counts take min(nshare, W) shares; the default schedule takes
    floor(sqrt(W)) (at most nshare), and for a batch whose nonzero lengths
    are all equal at most 256, aligned with its rows."""
    lens = [max(x, 0) for x in lens]
    W = sum(lens) * Hkv
    nz = [x for x in lens if x > 0]
    uniform = bool(nz) and min(nz) == max(nz)
    n = W
    if default:
        n = math.isqrt(W)
        if uniform:
            n = min(n, 256)
    n = max(1, min(nshare, n))
    if default and uniform:
        R, floor_n, best = len(nz) * Hkv, (4 * n + 4) // 5, 0
        if R <= n:
            best = R * (n // R)
        else:
            m, m_end = -(-R // n), -(-R // n) + 64
            while m < m_end and R // m >= floor_n:
                if R % m == 0:
                    best = R // m
                    break
                m += 1
        if best >= floor_n:
            n = best
    return n


def walk(lens, Hkv, n):
    """Items (share c, sequence b, kv head h, keys [k0, k1)) of every share."""
    lens = [max(x, 0) for x in lens]
    W = sum(lens) * Hkv
    P = [0]
    for x in lens:
        P.append(P[-1] + x)
    items = []
    for c in range(n):
        s, e = c * W // n, (c + 1) * W // n
        if s >= e:
            continue
        b = next(i for i in range(len(lens)) if P[i + 1] * Hkv > s)
        pos = s
        while pos < e:
            while pos >= (P[b] + lens[b]) * Hkv:
                b += 1
            off = pos - P[b] * Hkv
            h, k0 = divmod(off, lens[b])
            k1 = min(lens[b], k0 + (e - pos))
            items.append((c, b, h, k0, k1))
            pos += k1 - k0
    return items, W


def check(lens, Hkv, n):
    items, W = walk(lens, Hkv, n)
    B = len(lens)
    owner, slots, table = {}, set(), {}
    for c, b, h, k0, k1 in items:
        row = b * Hkv + h
        assert 0 <= h < Hkv and 0 <= k0 < k1 <= lens[b]
        for k in range(k0, k1):
            assert (row, k) not in owner
            owner[(row, k)] = c
        slot = c + row
        assert slot not in slots and slot < n + B * Hkv
        slots.add(slot)
        if k0 == 0:
            x_last = (sum(lens[:b]) * Hkv + h * lens[b]) + lens[b] - 1
            c_last = ((x_last + 1) * n - 1) // W
            table[row] = (c + row, c_last - c + 1)
    for b, L in enumerate(lens):
        for h in range(Hkv):
            row = b * Hkv + h
            assert all((row, k) in owner for k in range(max(L, 0)))
            if L > 0:
                first, count = table[row]
                holders = sorted({owner[(row, k)] for k in range(L)})
                assert holders == list(range(first - row, first - row + count))
    for x in range(0, W, max(1, W // 500)):
        c = ((x + 1) * n - 1) // W
        assert c * W // n <= x < (c + 1) * W // n


@pytest.mark.parametrize("seed", range(6))
def test_random_batches_explicit_share_counts(seed):
    rng = random.Random(seed)
    for _ in range(150):
        lens = [rng.choice([0, 1, 2, 15, 16, 17, rng.randint(0, 300)]) for _ in range(rng.randint(1, 10))]
        Hkv = rng.choice([1, 2, 3, 8])
        if sum(lens) == 0:
            continue
        n = share_count(lens, Hkv, rng.choice([1, 2, 3, 7, 64, 304]), False)
        check(lens, Hkv, n)


@pytest.mark.parametrize("seed", range(3))
def test_random_batches_default_schedule(seed):
    rng = random.Random(100 + seed)
    for _ in range(100):
        same = rng.random() < 0.5
        L0 = rng.randint(1, 3000)
        lens = [L0 if same else rng.randint(0, 3000) for _ in range(rng.randint(1, 12))]
        if same and rng.random() < 0.3:
            lens[0] = 0  # empty rows do not break uniformity
        Hkv = rng.choice([1, 2, 8])
        if sum(lens) == 0:
            continue
        n = share_count(lens, Hkv, 304, True)
        W = sum(lens) * Hkv
        assert 1 <= n <= 304
        assert n <= max(1, math.isqrt(W))  # the alignment never raises the count
        check(lens, Hkv, n)


@pytest.mark.parametrize("lens,Hkv,want", [
    ([8192] * 64, 8, 256),       # 512 rows: whole rows, two a share
    ([8192] * 128, 8, 256),      # 1024 rows: four a share
    ([8192] * 32, 8, 256),       # 256 rows: one a share
    ([32768] * 16, 8, 256),      # 128 rows cut in two
    ([8192] * 4, 8, 256),        # 32 rows cut in eight
    ([8192] * 2, 8, 256),        # 16 rows cut in sixteen
    ([8192], 8, 256),            # sqrt(65536) = 256 shares: 8 rows cut in 32
    ([512], 8, 64),              # sqrt(4096) = 64: 8 rows cut in 8
    ([2048], 8, 128),            # sqrt(16384) = 128: 8 rows cut in 16
    ([131072], 8, 256),          # 8 rows cut in 32
    ([40] * 64, 8, 128),         # 512 short rows: sqrt(20480) = 143, whole rows, 4 a share
    ([0, 100, 100, 0, 100], 2, 24),  # sqrt(600) = 24: 6 rows cut in 4
    ([16384, 131072, 50000], 8, 304),  # ragged: no cap, no alignment
])
def test_default_share_counts(lens, Hkv, want):
    assert share_count(lens, Hkv, 304, True) == want
