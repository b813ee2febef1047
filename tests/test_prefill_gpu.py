"""GPU prefill parity against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from parametrized_local_linear_gb300 import (PlxError, inputs, plx_check_device_error,
                                             plx_prefill_fwd, plx_prefill_fwd_f32)

from helpers import LSE_ABS, assert_bf16_close, assert_f32_close, device, sample_rows

pytestmark = pytest.mark.gpu


def _run(fn, q, k, v, r):
    dev = device()
    qd, kd, vd, rd = (t.to(dev) for t in (q, k, v, r))
    out = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device=dev)
    fn(qd, kd, vd, rd, out, lse)
    plx_check_device_error()
    return out.cpu(), lse.cpu()


# ------------------------------------------------------------------ fp32 path
def test_f32_tiny_workload_matches_oracle():
    w = inputs.TINY_PREFILL_F32
    q, k, v, r = inputs.prefill_inputs_for(w)
    out, lse = _run(plx_prefill_fwd_f32, q, k, v, r)
    ref, ref_lse = oracle.prefill(q, k, v, r)
    assert_f32_close(out.double().numpy(), ref, "out")
    assert_f32_close(lse.double().numpy(), ref_lse, "lse")


@pytest.mark.parametrize("B,Hq,Hkv,L,d", [(2, 4, 2, 77, 128), (1, 3, 1, 1, 64), (1, 2, 2, 130, 64)])
def test_f32_shapes_match_oracle(B, Hq, Hkv, L, d):
    q, k, v, r = inputs.prefill_inputs(B, Hq, Hkv, L, d, torch.float32, 0.1, 40 + L)
    out, lse = _run(plx_prefill_fwd_f32, q, k, v, r)
    ref, ref_lse = oracle.prefill(q, k, v, r)
    assert_f32_close(out.double().numpy(), ref, "out")
    assert_f32_close(lse.double().numpy(), ref_lse, "lse")


# ------------------------------------------------------------------ bf16 path
@pytest.mark.parametrize("B,Hq,Hkv,L", [
    (1, 2, 1, 256),    # two query tiles, eight key tiles
    (2, 4, 2, 200),    # ragged last query tile and key tile
    (1, 2, 2, 1),      # one row, one key
    (1, 1, 1, 64),     # exactly one key tile
    (1, 2, 1, 129),    # one row into the second query tile
    (1, 4, 1, 383),    # GQA group of 4, three query tiles, ragged
    (1, 8, 1, 300),    # GQA group of 8
    (1, 16, 1, 130),   # one kv head for 16 query heads (MQA), one-row tail
])
def test_bf16_small_matches_oracle_every_row(B, Hq, Hkv, L):
    q, k, v, r = inputs.prefill_inputs(B, Hq, Hkv, L, 128, torch.bfloat16, 0.05, 7 + L)
    out, lse = _run(plx_prefill_fwd, q, k, v, r)
    ref, ref_lse = oracle.prefill(q, k, v, r)
    assert_bf16_close(out.double().numpy(), ref, "out")
    np.testing.assert_allclose(lse.double().numpy(), ref_lse, rtol=0, atol=LSE_ABS)


def test_bf16_large_probe_and_values():
    """Larger probe (|r| ~ 0.5) and shifted values make the correction dominate."""
    q, k, v, r = inputs.prefill_inputs(1, 2, 1, 320, 128, torch.bfloat16, 0.5, 99)
    v = (v.float() + 3.0).to(torch.bfloat16)
    out, _ = _run(plx_prefill_fwd, q, k, v, r)
    ref, _ = oracle.prefill(q, k, v, r)
    assert_bf16_close(out.double().numpy(), ref, "out")


def test_bf16_rho_zero_is_softmax_attention():
    q, k, v, r = inputs.prefill_inputs(1, 4, 2, 300, 128, torch.bfloat16, 0.05, 5)
    out, lse = _run(plx_prefill_fwd, q, k, v, torch.zeros_like(r))
    kk = k.double().repeat_interleave(2, dim=1); vv = v.double().repeat_interleave(2, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), kk, vv, is_causal=True)
    assert_bf16_close(out.double().numpy(), ref.numpy(), "rho=0")


@pytest.mark.parametrize("w", [inputs.PREFILL_0P6B, inputs.PREFILL_1P7B], ids=lambda w: w.name)
def test_bf16_full_size_workload_sampled_rows(w):
    q, k, v, r = inputs.prefill_inputs_for(w)
    out, lse = _run(plx_prefill_fwd, q, k, v, r)
    rows = sample_rows(w.B, w.Hq, w.L, n_random=24, seed=w.seed)
    ref, ref_lse = oracle.prefill(q, k, v, r, rows=rows)
    idx = tuple(torch.as_tensor(a) for a in np.array(rows).T)
    got = out[idx].double().numpy()
    assert_bf16_close(got, ref, w.name)
    np.testing.assert_allclose(lse[idx].double().numpy(), ref_lse, rtol=0, atol=LSE_ABS)
    assert torch.isfinite(out).all(), "non-finite values in the full output"


def test_bf16_leaves_memory_outside_out_untouched():
    """Guard bands around out stay NaN: the TMA store clips to the tensor."""
    dev = device()
    q, k, v, r = inputs.prefill_inputs(1, 2, 1, 77, 128, torch.bfloat16, 0.05, 3)
    n = q.numel()
    buf = torch.full((n + 4096,), float("nan"), dtype=torch.bfloat16, device=dev)
    out = buf[2048:2048 + n].view_as(q)
    plx_prefill_fwd(q.to(dev), k.to(dev), v.to(dev), r.to(dev), out)
    plx_check_device_error()
    assert torch.isnan(buf[:2048]).all() and torch.isnan(buf[2048 + n:]).all()
    assert torch.isfinite(out).all()


def test_bf16_rejects_bad_head_dim():
    dev = device()
    q = torch.zeros(1, 2, 16, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(PlxError, match="head dim"):
        plx_prefill_fwd(q, q[:, :1].contiguous(), q[:, :1].contiguous(), q)


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk", [
    (1, 2, 1, 1, 300),      # a single new token over a cache
    (2, 4, 2, 77, 333),     # offset not a multiple of the tile sizes
    (1, 2, 2, 200, 200),    # Lq == Lk: plain prefill
    (1, 4, 2, 129, 1000),   # a chunk just over one query tile
])
def test_bf16_chunked_prefill_matches_oracle(B, Hq, Hkv, Lq, Lk):
    from parametrized_local_linear_gb300 import plx_prefill_fwd_chunk
    dev = device()
    q, k, v, r = inputs.prefill_inputs(B, Hq, Hkv, Lk, 128, torch.bfloat16, 0.05, Lq + Lk)
    qc, rc = q[:, :, -Lq:].contiguous(), r[:, :, -Lq:].contiguous()
    out = torch.full(qc.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full(qc.shape[:3], float("nan"), device=dev)
    plx_prefill_fwd_chunk(qc.to(dev), k.to(dev), v.to(dev), rc.to(dev), out, lse)
    plx_check_device_error()
    ref, ref_lse = oracle.prefill(qc, k, v, rc)
    assert_bf16_close(out.double().cpu().numpy(), ref, "chunk")
    np.testing.assert_allclose(lse.double().cpu().numpy(), ref_lse, rtol=0, atol=LSE_ABS)


def test_bf16_chunk_equals_tail_of_full_prefill_on_gpu():
    from parametrized_local_linear_gb300 import plx_prefill_fwd_chunk
    dev = device()
    q, k, v, r = (t.to(dev) for t in inputs.prefill_inputs(2, 4, 2, 700, 128, torch.bfloat16, 0.05, 8))
    full, _ = plx_prefill_fwd(q, k, v, r)
    part, _ = plx_prefill_fwd_chunk(q[:, :, 500:].contiguous(), k, v, r[:, :, 500:].contiguous())
    plx_check_device_error()
    # Same keys, same tiles, same arithmetic per row: bit-identical.
    assert torch.equal(part, full[:, :, 500:])


def test_chunk_rejects_lq_above_lk():
    from parametrized_local_linear_gb300 import plx_prefill_fwd_chunk
    dev = device()
    q = torch.zeros(1, 2, 64, 128, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 1, 32, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(PlxError, match="Lk"):
        plx_prefill_fwd_chunk(q, k, k, q)


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk", [
    (1, 2, 1, 300, 300),    # plain prefill, ragged last tile
    (2, 4, 2, 77, 333),     # chunk, offset not a multiple of the tile sizes
    (1, 4, 2, 129, 1000),   # chunk just over one query tile
])
def test_bf16_cor_matches_oracle(B, Hq, Hkv, Lq, Lk):
    from parametrized_local_linear_gb300 import plx_prefill_fwd_chunk, plx_prefill_fwd_cor
    from helpers import assert_cor_close, cor_bounds_prefill
    dev = device()
    q, k, v, r = inputs.prefill_inputs(B, Hq, Hkv, Lk, 128, torch.bfloat16, 0.05, 3 * Lq + Lk)
    qc, rc = q[:, :, -Lq:].contiguous().to(dev), r[:, :, -Lq:].contiguous().to(dev)
    kd, vd = k.to(dev), v.to(dev)
    cor = torch.full(qc.shape[:3], float("nan"), device=dev)
    out, _, _ = plx_prefill_fwd_cor(qc, kd, vd, rc, cor=cor)
    plain, _ = plx_prefill_fwd_chunk(qc, kd, vd, rc)
    plx_check_device_error()
    # The side output leaves o untouched.
    assert torch.equal(out, plain)
    _, _, ref = oracle.prefill(qc.cpu(), k, v, rc.cpu(), with_cor=True)
    assert_cor_close(cor.cpu().numpy(), ref, cor_bounds_prefill(qc.cpu(), k, v, rc.cpu()),
                     "prefill cor")


def test_bf16_cor_full_size_sampled_rows():
    """The 0.6B-shaped workload in the launch configuration the benchmark
    times, ratio checked on sampled rows against the explicit-Sigma oracle."""
    from parametrized_local_linear_gb300 import plx_prefill_fwd_cor
    from helpers import assert_cor_close, cor_bounds_prefill, sample_rows
    dev = device()
    w = inputs.PREFILL_0P6B
    q, k, v, r = inputs.prefill_inputs_for(w)
    _, _, cor = plx_prefill_fwd_cor(*(t.to(dev) for t in (q, k, v, r)))
    plx_check_device_error()
    rows = sample_rows(w.B, w.Hq, w.L, 40, 77)
    _, _, ref = oracle.prefill(q, k, v, r, rows=rows, with_cor=True)
    got = cor.cpu().numpy()[tuple(np.array(rows).T)]
    assert_cor_close(got, ref, cor_bounds_prefill(q, k, v, r, rows=rows), "prefill cor, full size")
