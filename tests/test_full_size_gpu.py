"""Full-coverage parity at the model-sized workloads, in the launch
configuration the benchmark times: every output row of the GPU prefill, every
(sequence, head) of the GPU decode and every row and key of the GPU backward
against the expanded fp64 oracle (dense O1 - O2 + O1*s and its closed-form
gradient), which the CPU tests pin to the explicit-Sigma oracle. The sampled
explicit-Sigma checks in the other test files remain the second anchor.

The prefill shape B=8, L=1024 has 1024 work items of 128 query rows for the
persistent kernel's one CTA per SM, so every CTA runs several items in a row
(TMEM, barrier phases and the epilogue hand-off carried across items), and
each of those items is checked on every row."""
import numpy as np
import pytest
import torch

from oracle import expanded
from parametrized_local_linear_gb300 import (inputs, plx_check_device_error, plx_decode_fwd,
                                             plx_decode_fwd_cor, plx_prefill_bwd, plx_prefill_fwd,
                                             plx_prefill_fwd_chunk, plx_prefill_fwd_cor,
                                             plx_prefill_fwd_train)

from helpers import (LSE_ABS, SBAR_ABS, assert_bf16_close, assert_cor_close, assert_grad_close,
                     cor_bounds_decode, cor_bounds_prefill, device)

pytestmark = pytest.mark.gpu

MULTI_ITEM = inputs.PrefillShape("prefill_multi_item_B8_Hq16_Hkv8_L1024_d128", 8, 16, 8, 1024,
                                 128, torch.bfloat16, 0.05, 1011)


def _lse_close(got, ref, what):
    err = float(np.max(np.abs(got - ref)))
    print(f"{what}: max|lse err| = {err:.2e}")
    assert err <= LSE_ABS, f"{what}: max|lse err| {err:.3e} > {LSE_ABS}"


@pytest.mark.parametrize("w", [inputs.PREFILL_0P6B, inputs.PREFILL_1P7B, MULTI_ITEM],
                         ids=lambda w: w.name)
def test_prefill_every_row(w):
    dev = device()
    q, k, v, r = inputs.prefill_inputs_for(w)
    if w is MULTI_ITEM:
        assert w.B * w.Hq * (w.L // 128) >= 6 * torch.cuda.get_device_properties(0).multi_processor_count
    qd, kd, vd, rd = (t.to(dev) for t in (q, k, v, r))
    out = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device=dev)
    plx_prefill_fwd(qd, kd, vd, rd, out, lse)
    plx_check_device_error()
    ref, ref_lse = expanded.prefill(q, k, v, r)
    err, bound = assert_bf16_close(out.double().cpu().numpy(), ref, w.name)
    print(f"{w.name}: max|err| {err:.3e} (bound {bound:.3e})")
    _lse_close(lse.double().cpu().numpy(), ref_lse, w.name)


def test_chunk_every_row():
    """The chunk the benchmark times: the last 2048 of 16384 positions,
    1.7B-shaped heads."""
    dev = device()
    w = inputs.PREFILL_1P7B
    q, k, v, r = inputs.prefill_inputs_for(w)
    qc, rc = q[:, :, -2048:].contiguous(), r[:, :, -2048:].contiguous()
    out, lse = plx_prefill_fwd_chunk(qc.to(dev), k.to(dev), v.to(dev), rc.to(dev),
                                     lse=torch.empty(qc.shape[:3], device=dev))
    plx_check_device_error()
    ref, ref_lse = expanded.prefill(qc, k, v, rc)
    assert_bf16_close(out.double().cpu().numpy(), ref, "chunk 2048 of 16384")
    _lse_close(lse.double().cpu().numpy(), ref_lse, "chunk 2048 of 16384")


def test_training_forward_and_cor_every_row():
    """o^SA and sbar of the training forward, and the COR side output, on every
    row of the 0.6B-shaped workload."""
    dev = device()
    w = inputs.PREFILL_0P6B
    q, k, v, r = inputs.prefill_inputs_for(w)
    qd, kd, vd, rd = (t.to(dev) for t in (q, k, v, r))
    out, lse, o1, sbar = plx_prefill_fwd_train(qd, kd, vd, rd)
    _, _, cor = plx_prefill_fwd_cor(qd, kd, vd, rd)
    plx_check_device_error()
    ref, _, ref_osa, ref_sbar, ref_cor = expanded.prefill(q, k, v, r, with_parts=True)
    assert_bf16_close(out.double().cpu().numpy(), ref, "train forward o")
    assert_bf16_close(o1.double().cpu().numpy(), ref_osa, "train forward o^SA")
    serr = float(np.max(np.abs(sbar.double().cpu().numpy() - ref_sbar)))
    assert serr <= SBAR_ABS, f"sbar: {serr:.3e} > {SBAR_ABS}"
    assert_cor_close(cor.cpu().numpy(), ref_cor, cor_bounds_prefill(q, k, v, r),
                     "prefill cor, every row")


@pytest.mark.parametrize("w", [inputs.DECODE_B64, inputs.DECODE_RAGGED], ids=lambda w: w.name)
def test_decode_every_pair(w):
    dev = device()
    q, r, kc, vc, sl = inputs.decode_inputs_for(w)
    qd, rd, kd, vd, sd = (t.to(dev) for t in (q, r, kc, vc, sl))
    out = plx_decode_fwd(qd, rd, kd, vd, sd, torch.full_like(qd, float("nan")))
    _, cor = plx_decode_fwd_cor(qd, rd, kd, vd, sd)
    plx_check_device_error()
    ref, _, ref_cor = expanded.decode(q, r, kc, vc, sl, with_cor=True)
    err, bound = assert_bf16_close(out.double().cpu().numpy(), ref, w.name)
    print(f"{w.name}: max|err| {err:.3e} (bound {bound:.3e})")
    assert_cor_close(cor.cpu().numpy(), ref_cor, cor_bounds_decode(q, r, kc, vc, sl),
                     w.name + " cor")


@pytest.mark.parametrize("w", [inputs.PREFILL_0P6B, inputs.PREFILL_1P7B], ids=lambda w: w.name)
def test_backward_every_row_and_key(w):
    dev = device()
    q, k, v, r = inputs.prefill_inputs_for(w)
    g = torch.Generator().manual_seed(w.seed + 7)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    qd, kd, vd, rd, dod = (t.to(dev) for t in (q, k, v, r, do))
    o, lse, o1, sb = plx_prefill_fwd_train(qd, kd, vd, rd)
    fill = lambda t: torch.full_like(t, float("nan"))  # noqa: E731
    got = plx_prefill_bwd(qd, kd, vd, rd, o, o1, lse, sb, dod, fill(qd), fill(kd), fill(vd),
                          fill(rd))
    plx_check_device_error()
    want = expanded.prefill_grad(q, k, v, r, do)
    for name, g_, w_ in zip(("dq", "dk", "dv", "dr"), got, want):
        assert_grad_close(g_.double().cpu().numpy(), w_, f"{name} {w.name}")
