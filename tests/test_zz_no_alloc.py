"""The allocation-free decode entry point (plx_decode_fwd_noalloc).

Some callers cannot allocate device memory while they call into this
library; this entry point serves them by keeping its partial records in a fixed
device array. It must give the same result as plx_decode_fwd, call after
call, because the array is reused and keeps the previous call's contents.
This file is named so that pytest collects it last."""
import ctypes

import pytest
import torch

from parametrized_local_linear_gb300 import binding, inputs, plx_check_device_error, plx_decode_fwd

from helpers import BF16_ABS, BF16_REL, device

pytestmark = pytest.mark.gpu


def _call_noalloc(q, r, kc, vc, sl, out):
    L = binding.lib()
    B, Hq, d = q.shape
    st = L.plx_decode_fwd_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(r.data_ptr()),
                                  ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
                                  ctypes.c_void_p(sl.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                  B, Hq, kc.shape[1], d,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == binding.PLX_OK, binding.lib().plx_last_error_message()


@pytest.mark.parametrize("lens,Hq,Hkv", [
    ([1, 5, 33, 0, 200, 64], 4, 2),      # an empty sequence, a one-token one, sub-tile lengths
    ([300, 301], 8, 1),                  # 8 query heads a kv head
    ([3000, 17, 12000], 16, 8),          # rows cut between several CTAs
])
def test_noalloc_decode_matches_the_oracle(lens, Hq, Hkv):
    """The allocation-free decode against the fp64 oracle directly, not only
    against the allocating entry point."""
    import oracle
    from helpers import assert_bf16_close
    dev = device()
    q, r, kc, vc, sl = inputs.decode_inputs(len(lens), Hq, Hkv, 128, lens, torch.bfloat16, 0.05,
                                            5 + len(lens))
    qd, rd, kd, vd, sd = (t.to(dev) for t in (q, r, kc, vc, sl))
    out = torch.full_like(qd, float("nan"))
    _call_noalloc(qd, rd, kd, vd, sd, out)
    plx_check_device_error()
    ref, _ = oracle.decode(q, r, kc, vc, sl)
    assert_bf16_close(out.double().cpu().numpy(), ref, f"no-alloc decode {lens}")


def test_noalloc_decode_matches_allocating_decode_twice():
    dev = device()
    cases = [([700, 0, 33, 4100], 16, 8, 21), ([9000, 130], 4, 2, 22)]
    for lens, Hq, Hkv, seed in cases:  # two calls in a row, different shapes
        q, r, kc, vc, sl = (t.to(dev) for t in inputs.decode_inputs(
            len(lens), Hq, Hkv, 128, lens, torch.bfloat16, 0.05, seed))
        ref = plx_decode_fwd(q, r, kc, vc, sl)
        out = torch.full_like(q, float("nan"))
        _call_noalloc(q, r, kc, vc, sl, out)
        plx_check_device_error()
        ref_f, out_f = ref.float(), out.float()
        assert torch.isfinite(out_f).all()
        err = (out_f - ref_f).abs().max().item()
        assert err <= BF16_REL * ref_f.abs().max().item() + BF16_ABS, err


def test_noalloc_decode_rejects_too_many_records():
    device()
    z = torch.zeros(16, device="cuda", dtype=torch.bfloat16)
    p = ctypes.c_void_p(z.data_ptr())
    # the row table plus B * Hq records of (2 * 128 + 2) * 4 bytes > 16 MiB even with one share
    st = binding.lib().plx_decode_fwd_noalloc(p, p, p, p, p, p, 8192, 8, 8, 128, None)
    assert st == binding.PLX_ERR_UNSUPPORTED
    assert b"fixed array" in binding.lib().plx_last_error_message()
