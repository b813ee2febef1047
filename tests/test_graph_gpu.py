"""The C-ABI calls are stream-ordered with no host synchronisation, so whole
steps can be captured into a CUDA graph and replayed (the stream-ordered
workspace allocations become graph memory nodes). Replays must reproduce the
eager results bit for bit."""
import pytest
import torch

from parametrized_local_linear_gb300 import (inputs, plx_check_device_error, plx_decode_fwd,
                                             plx_prefill_bwd, plx_prefill_fwd_train, plx_qkvr_proj)

from helpers import device

pytestmark = pytest.mark.gpu


def test_training_step_replays_in_a_cuda_graph():
    dev = device()
    B, L, D, Hq, Hkv, d = 2, 200, 256, 2, 1, 128
    g = torch.Generator().manual_seed(31)
    x = torch.randn(B * L, D, generator=g).to(torch.bfloat16).to(dev)
    w = (torch.randn((2 * Hq + 2 * Hkv) * d, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    w[(Hq + 2 * Hkv) * d:] *= 0.05
    w = w.to(dev)
    do = torch.randn(B, Hq, L, d, generator=g).to(torch.bfloat16).to(dev)
    qh = torch.empty(B, Hq, L, d, dtype=torch.bfloat16, device=dev)
    kh = torch.empty(B, Hkv, L, d, dtype=torch.bfloat16, device=dev)
    vh, rh = torch.empty_like(kh), torch.empty_like(qh)
    out, o1 = torch.empty_like(qh), torch.empty_like(qh)
    lse = torch.empty(B, Hq, L, device=dev)
    sb = torch.empty_like(lse)
    grads = [torch.empty_like(t) for t in (qh, kh, vh, rh)]

    def step():
        plx_qkvr_proj(x, w, B, L, Hq, Hkv, d, q=qh, k=kh, v=vh, r=rh)
        plx_prefill_fwd_train(qh, kh, vh, rh, out, lse, o1, sb)
        plx_prefill_bwd(qh, kh, vh, rh, out, o1, lse, sb, do, *grads)

    step()  # eager, and the first call on the device (before any capture)
    torch.cuda.synchronize()
    plx_check_device_error()
    want = [t.clone() for t in [out, lse] + grads]
    for t in [out, lse] + grads:
        t.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    plx_check_device_error()
    for a, b in zip([out, lse] + grads, want):
        assert torch.equal(a, b)


def test_decode_replays_in_a_cuda_graph():
    dev = device()
    lens = [5, 0, 1000, 333]
    q, r, kc, vc, sl = (t.to(dev) for t in inputs.decode_inputs(len(lens), 4, 2, 128, lens,
                                                                 torch.bfloat16, 0.05, 32))
    out = torch.empty_like(q)
    plx_decode_fwd(q, r, kc, vc, sl, out)
    torch.cuda.synchronize()
    want = out.clone()
    out.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        plx_decode_fwd(q, r, kc, vc, sl, out)
    graph.replay()
    torch.cuda.synchronize()
    plx_check_device_error()
    assert torch.equal(out, want)
