"""The debug build (PLX_DEBUG_BOUNDS: device-side index checks before every
TMA copy and indexed store, see include/plx.h) on valid inputs: every entry
point reports no failed check, and its outputs equal the release library's
bit for bit, so the checks change nothing but the reporting."""
import ctypes

import pytest
import torch

from parametrized_local_linear_gb300 import (binding, inputs, plx_check_device_error,
                                             plx_decode_fwd, plx_decode_fwd_cor, plx_prefill_bwd,
                                             plx_prefill_fwd, plx_prefill_fwd_chunk,
                                             plx_prefill_fwd_train, plx_qkvr_proj)

from helpers import device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    device()
    return binding.load_debug_lib()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ok(dbg, status):
    assert status == binding.PLX_OK, dbg.plx_last_error_message()
    st = dbg.plx_check_device_error(_s())
    assert st == binding.PLX_OK, dbg.plx_last_error_message()


def test_debug_prefill_chunk_train_backward(dbg):
    dev = device()
    q, k, v, r = (t.to(dev) for t in inputs.prefill_inputs(2, 4, 2, 200, 128, torch.bfloat16,
                                                            0.05, 17))
    B, Hq, L, d = q.shape
    out, lse = torch.empty_like(q), torch.empty(q.shape[:3], device=dev)
    _ok(dbg, dbg.plx_prefill_fwd(_p(q), _p(k), _p(v), _p(r), _p(out), _p(lse), B, Hq, 2, L, d, _s()))
    ref, ref_lse = plx_prefill_fwd(q, k, v, r, lse=torch.empty_like(lse))
    plx_check_device_error()
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    qc, rc = q[:, :, 123:].contiguous(), r[:, :, 123:].contiguous()
    oc = torch.empty_like(qc)
    _ok(dbg, dbg.plx_prefill_fwd_chunk(_p(qc), _p(k), _p(v), _p(rc), _p(oc), None, B, Hq, 2,
                                       L - 123, L, d, _s()))
    assert torch.equal(oc, plx_prefill_fwd_chunk(qc, k, v, rc)[0])
    o, l, o1, sb = (torch.empty_like(x) for x in plx_prefill_fwd_train(q, k, v, r))
    _ok(dbg, dbg.plx_prefill_fwd_train(_p(q), _p(k), _p(v), _p(r), _p(o), _p(l), _p(o1), _p(sb),
                                       B, Hq, 2, L, d, _s()))
    ro, rl, ro1, rsb = plx_prefill_fwd_train(q, k, v, r)
    assert all(torch.equal(x, y) for x, y in ((o, ro), (l, rl), (o1, ro1), (sb, rsb)))
    do = torch.randn(q.shape, device=dev).to(torch.bfloat16)
    g = [torch.empty_like(x) for x in (q, k, v, r)]
    _ok(dbg, dbg.plx_prefill_bwd(*(_p(x) for x in (q, k, v, r, o, o1, l, sb, do, *g)),
                                 B, Hq, 2, L, d, _s()))
    want = plx_prefill_bwd(q, k, v, r, o, o1, l, sb, do)
    plx_check_device_error()
    assert all(torch.equal(x, y) for x, y in zip(g, want))


def test_debug_projection(dbg):
    dev = device()
    B, L, D, Hq, Hkv = 1, 300, 256, 2, 1
    x = torch.randn(B * L, D, device=dev).to(torch.bfloat16)
    w = (torch.randn((2 * Hq + 2 * Hkv) * 128, D, device=dev) / 16).to(torch.bfloat16)
    ref = plx_qkvr_proj(x, w, B, L, Hq, Hkv)
    outs = [torch.empty_like(t) for t in ref]
    _ok(dbg, dbg.plx_qkvr_proj(_p(x), _p(w), *(_p(t) for t in outs), B, L, D, Hq, Hkv, 128, _s()))
    assert all(torch.equal(a, b) for a, b in zip(outs, ref))


@pytest.mark.parametrize("lens,nsplit", [([700, 0, 33, 4100, 5], 0), ([17, 1, 33], 500),
                                         ([3], 0), ([0, 0], 3)])
def test_debug_decode(dbg, lens, nsplit):
    dev = device()
    q, r, kc, vc, sl = (t.to(dev) for t in inputs.decode_inputs(
        len(lens), 16, 8, 128, lens, torch.bfloat16, 0.05, 9 + len(lens)))
    if kc.shape[0] == 0:
        kc = torch.zeros(16, 8, 128, dtype=torch.bfloat16, device=dev)
        vc = kc.clone()
    B = len(lens)
    out = torch.empty_like(q)
    nbytes = binding.lib().plx_decode_workspace_bytes(B, 16, 8, 128, max(nsplit, 1) if nsplit else
                                                      binding.lib().plx_decode_default_nsplit(B, 8))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _ok(dbg, dbg.plx_decode_fwd_ex(_p(q), _p(r), _p(kc), _p(vc), _p(sl), _p(out), B, 16, 8, 128,
                                   nsplit, _p(ws), nbytes, _s()))
    assert torch.equal(out, plx_decode_fwd(q, r, kc, vc, sl, nsplit=nsplit, workspace=ws))
    cor = torch.empty(B, 16, device=dev)
    _ok(dbg, dbg.plx_decode_fwd_cor(_p(q), _p(r), _p(kc), _p(vc), _p(sl), _p(out), _p(cor), B, 16,
                                    8, 128, _s()))
    ro, rc = plx_decode_fwd_cor(q, r, kc, vc, sl)
    plx_check_device_error()
    assert torch.equal(out, ro) and torch.equal(cor, rc)
