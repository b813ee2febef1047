"""Bounded waits: a wait that runs out reports an error status and leaves the
GPU usable. The failure is a flag that nothing sets (an mbarrier no thread
arrives on), never a fault, trap or endless loop."""
import pytest
import torch

from parametrized_local_linear_gb300 import (PlxError, binding, inputs, plx_check_device_error,
                                             plx_debug_timeout_probe, plx_prefill_fwd)

from helpers import device

pytestmark = pytest.mark.gpu


def test_timed_out_wait_is_reported_and_context_survives():
    dev = device()
    plx_check_device_error()  # start clean
    plx_debug_timeout_probe(limit_cycles=200000)
    with pytest.raises(PlxError) as ei:
        plx_check_device_error()
    assert ei.value.status == binding.PLX_ERR_DEVICE_TIMEOUT
    plx_check_device_error()  # the word was cleared
    # The context still runs real work.
    q, k, v, r = inputs.prefill_inputs(1, 2, 1, 64, 128, torch.bfloat16, 0.05, 1)
    out, _ = plx_prefill_fwd(*(t.to(dev) for t in (q, k, v, r)))
    plx_check_device_error()
    assert torch.isfinite(out).all()
