"""GPU decode (equal shares of the batch's key stream + log-sum-exp combine)
parity against the fp64 oracle."""
import random

import numpy as np
import pytest
import torch

import oracle
from parametrized_local_linear_gb300 import (inputs, plx_check_device_error,
                                             plx_decode_default_nsplit, plx_decode_fwd,
                                             plx_decode_workspace_bytes, plx_prefill_fwd)

from helpers import assert_bf16_close, device

pytestmark = pytest.mark.gpu


def _to(dev, *ts):
    return [t.to(dev) for t in ts]


def _decode(q, r, kc, vc, sl, **kw):
    dev = device()
    qd, rd, kd, vd, sd = _to(dev, q, r, kc, vc, sl)
    out = torch.full_like(qd, float("nan"))
    plx_decode_fwd(qd, rd, kd, vd, sd, out, **kw)
    plx_check_device_error()
    return out.cpu()


@pytest.mark.parametrize("lens,Hq,Hkv", [
    ([1, 5, 33, 0, 200, 64], 4, 2),      # includes an empty sequence and sub-tile lengths
    ([1000, 17, 4096], 16, 8),           # model head layout
    ([300, 301], 8, 1),                  # GQA group of 8
])
def test_decode_matches_oracle_all_pairs(lens, Hq, Hkv):
    q, r, kc, vc, sl = inputs.decode_inputs(len(lens), Hq, Hkv, 128, lens, torch.bfloat16, 0.05,
                                            len(lens) + Hq)
    out = _decode(q, r, kc, vc, sl)
    ref, _ = oracle.decode(q, r, kc, vc, sl)
    assert_bf16_close(out.double().numpy(), ref, "decode")
    for b, n in enumerate(lens):
        if n == 0:
            assert torch.all(out[b] == 0)


def _share_invariance_bound(q, r, kc, vc, lens, base):
    """Per-element bound on |o(n1) - o(n2)| between two share counts.

    A share count moves the running max each CTA exponentiates against, and
    so the bf16 rounding of every weight p_j and product p_j t_j that enters
    the value products (relative error at most 2^-8 each, for either run:
    bf16 keeps 8 significant bits, rounded to nearest).
    With w the normalised weights, t_j = rho . k_j and s = sum_j w_j t_j, one
    run's O1 = sum w v and O2 = sum w t v then move by at most
    2^-8 sum_j w_j |v_j| and 2^-8 sum_j w_j |t_j v_j| per element, and
    o = O1 (1 + s) - O2 by at most 2^-8 ((1 + |s|) sum w |v| + sum w |t v|);
    two runs double that. Each output is rounded to bf16 once (half an ulp
    each, one ulp together); fp32 summation order adds far less."""
    B, Hq, d = q.shape
    G = Hq // kc.shape[1]
    offs = np.concatenate([[0], np.cumsum(lens)])
    bound = np.zeros((B, Hq, d))
    for b in range(B):
        K = kc[offs[b]:offs[b + 1]].double()
        V = vc[offs[b]:offs[b + 1]].double()
        for h in range(Hq):
            Kh, Vh = K[:, h // G], V[:, h // G]
            w = torch.softmax(Kh @ q[b, h].double() / np.sqrt(d), dim=0)
            t = Kh @ r[b, h].double()
            s = float((w * t).sum())
            bound[b, h] = 2 * 2.0 ** -8 * ((1 + abs(s)) * (w @ Vh.abs()) + w @ (t.abs()[:, None] * Vh.abs())).numpy()
    mag = np.abs(base.double().numpy())
    ulp = np.where(mag > 0, 2.0 ** (np.floor(np.log2(np.where(mag > 0, mag, 1.0))) - 7), 2.0 ** -133)
    return bound + ulp


@pytest.mark.parametrize("nsplit", [1, 3, 7, 64, 2000])
def test_decode_share_count_does_not_change_the_result(nsplit):
    lens = [700, 1, 129, 2048]
    q, r, kc, vc, sl = inputs.decode_inputs(len(lens), 16, 8, 128, lens, torch.bfloat16, 0.05, 77)
    base = _decode(q, r, kc, vc, sl, nsplit=1).float()
    out = _decode(q, r, kc, vc, sl, nsplit=nsplit).float()
    bound = _share_invariance_bound(q, r, kc, vc, lens, base)
    diff = torch.abs(out - base).double().numpy()
    worst = float(np.max(diff / bound))
    print(f"nsplit {nsplit}: max |diff| / bound = {worst:.3f}, max |diff| = {diff.max():.2e}")
    assert worst <= 1.0, f"share count {nsplit}: a difference exceeds its bound ({worst:.2f}x)"


def test_decode_with_caller_workspace():
    dev = device()
    lens = [90, 4000]
    q, r, kc, vc, sl = inputs.decode_inputs(2, 4, 2, 128, lens, torch.bfloat16, 0.05, 8)
    nsplit = 5
    nbytes = plx_decode_workspace_bytes(2, 4, 2, 128, nsplit)
    ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device=dev)
    out = _decode(q, r, kc, vc, sl, nsplit=nsplit, workspace=ws)
    ref, _ = oracle.decode(q, r, kc, vc, sl)
    assert_bf16_close(out.double().numpy(), ref, "decode+workspace")


def test_decode_equals_last_prefill_row_on_gpu():
    """Decode over a cache equals the last row of a prefill over the same keys."""
    dev = device()
    L, Hq, Hkv = 333, 4, 2
    q, k, v, r = inputs.prefill_inputs(1, Hq, Hkv, L, 128, torch.bfloat16, 0.05, 12)
    pre, _ = plx_prefill_fwd(*_to(dev, q, k, v, r))
    kc = k[0].permute(1, 0, 2).contiguous()  # [L, Hkv, d]
    vc = v[0].permute(1, 0, 2).contiguous()
    out = _decode(q[:, :, -1].contiguous(), r[:, :, -1].contiguous(), kc, vc,
                  torch.tensor([L], dtype=torch.int32))
    assert_bf16_close(out[0].double().numpy(), pre[0, :, -1].double().cpu().numpy(), "decode-vs-prefill")


@pytest.mark.parametrize("w", [inputs.DECODE_B64, inputs.DECODE_RAGGED], ids=lambda w: w.name)
def test_decode_full_size_workload_sampled_pairs(w):
    q, r, kc, vc, sl = inputs.decode_inputs_for(w)
    out = _decode(q, r, kc, vc, sl)
    rng = random.Random(w.seed)
    pairs = sorted({(0, 0), (w.B - 1, w.Hq - 1)} |
                   {(rng.randrange(w.B), rng.randrange(w.Hq)) for _ in range(10)})
    ref, _ = oracle.decode(q, r, kc, vc, sl, pairs=pairs, threads=8)
    got = np.stack([out[b, h].double().numpy() for b, h in pairs])
    assert_bf16_close(got, ref, w.name)
    assert torch.isfinite(out).all()


def test_default_share_count_is_sane():
    device()
    n = plx_decode_default_nsplit(64, 8)
    # Two CTAs per SM, whatever the batch.
    assert n == 2 * torch.cuda.get_device_properties(0).multi_processor_count
    assert plx_decode_default_nsplit(1, 1) == n


@pytest.mark.parametrize("lens,Hq,Hkv,nsplit", [
    ([0, 0, 5, 0, 300, 0], 4, 2, 7),     # empty sequences before, between and after
    ([1] * 40, 8, 1, 3),                 # one-key sequences: a share holds many rows
    ([17, 1, 33], 16, 8, 500),           # more shares than keys: one key a share
    ([2048, 0, 4095], 2, 1, 64),         # shares cut long rows at tile-unaligned keys
    ([100], 16, 8, 0),                   # default schedule, 800 keys: 2 shares of 400
    ([3, 700, 9, 1500], 8, 4, 0),        # default schedule across ragged rows
    ([40] * 64, 16, 8, 0),               # default, one length: 32 shares of 16 whole rows
    ([0, 100, 100, 0, 100], 4, 2, 0),    # default, one length among empty rows: 3 rows a share
])
def test_decode_shares_across_rows(lens, Hq, Hkv, nsplit):
    """The batch's keys are one stream cut into equal shares; shares start and
    end inside rows, hold several rows, or hold a single key."""
    q, r, kc, vc, sl = inputs.decode_inputs(len(lens), Hq, Hkv, 128, lens, torch.bfloat16, 0.05,
                                            3 * len(lens) + nsplit)
    out = _decode(q, r, kc, vc, sl, nsplit=nsplit)
    ref, _ = oracle.decode(q, r, kc, vc, sl)
    assert_bf16_close(out.double().numpy(), ref, f"decode shares {lens} nsplit {nsplit}")
    for b, n in enumerate(lens):
        if n == 0:
            assert torch.all(out[b] == 0)


def test_decode_all_sequences_empty():
    lens = [0, 0, 0]
    q, r, kc, vc, sl = inputs.decode_inputs(3, 4, 2, 128, lens, torch.bfloat16, 0.05, 5)
    kc = torch.zeros(16, 2, 128, dtype=torch.bfloat16)  # a cache holding no sequence's keys
    vc = torch.zeros_like(kc)
    for nsplit in (0, 1, 9):
        out = _decode(q, r, kc, vc, sl, nsplit=nsplit)
        assert torch.all(out == 0)


@pytest.mark.parametrize("lens,Hq,Hkv", [
    ([1, 5, 33, 0, 200, 64], 4, 2),      # an empty sequence, a one-token one, sub-tile lengths
    ([1000, 17, 4096], 16, 8),           # model head layout
])
def test_decode_cor_matches_oracle(lens, Hq, Hkv):
    from parametrized_local_linear_gb300 import plx_decode_fwd_cor
    from helpers import assert_cor_close, cor_bounds_decode
    dev = device()
    q, r, kc, vc, sl = inputs.decode_inputs(len(lens), Hq, Hkv, 128, lens, torch.bfloat16, 0.05,
                                            2 * len(lens) + Hq)
    qd, rd, kd, vd, sd = _to(dev, q, r, kc, vc, sl)
    cor = torch.full((len(lens), Hq), float("nan"), device=dev)
    out, _ = plx_decode_fwd_cor(qd, rd, kd, vd, sd, cor=cor)
    plain = plx_decode_fwd(qd, rd, kd, vd, sd)
    plx_check_device_error()
    assert torch.equal(out, plain)  # the side output leaves o untouched
    _, _, ref = oracle.decode(q, r, kc, vc, sl, with_cor=True)
    assert_cor_close(cor.cpu().numpy(), ref, cor_bounds_decode(q, r, kc, vc, sl), "decode cor")
    for b, n in enumerate(lens):
        if n == 0:
            assert torch.all(cor[b] == 0)  # no keys: o = 0 and the ratio is defined as 0


def test_decode_lengths_past_the_token_extent_are_reported():
    """Lengths are on the device, so the host cannot check their sum; a batch
    whose lengths sum to 2^30 tokens or more (past the cache maps' extent) does
    no work and is reported by plx_check_device_error, and the next call runs
    normally. The cache is never read in that call, so a small one stands in."""
    from parametrized_local_linear_gb300 import PlxError, binding
    dev = device()
    q, r, kc, vc, _ = inputs.decode_inputs(2, 4, 2, 128, [16, 16], torch.bfloat16, 0.05, 3)
    qd, rd, kd, vd = _to(dev, q, r, kc, vc)
    big = torch.tensor([1 << 29, 1 << 29], dtype=torch.int32, device=dev)
    out = torch.empty_like(qd)
    plx_decode_fwd(qd, rd, kd, vd, big, out)
    with pytest.raises(PlxError) as exc:
        plx_check_device_error()
    assert exc.value.status == binding.PLX_ERR_INVALID_ARG
    # The error word was cleared; an ordinary call on the same device works.
    sl = torch.tensor([16, 16], dtype=torch.int32)
    got = _decode(q, r, kc, vc, sl)
    ref, _ = oracle.decode(q, r, kc, vc, sl)
    assert_bf16_close(got.double().numpy(), ref, "decode after a reported error")
