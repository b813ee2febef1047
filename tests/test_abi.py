"""The C-ABI library loads and exports every entry point include/plx.h
declares, and its host-side argument checks reject bad calls before any CUDA
call is made (CPU only: nothing here launches a kernel)."""
import ctypes
import os
import re

import pytest

from parametrized_local_linear_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "plx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(plx_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("plx_prefill_fwd", "plx_prefill_fwd_f32", "plx_decode_fwd", "plx_status_string"):
        assert s in syms


def test_every_declared_symbol_is_exported(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), s
        assert s in binding.SIGNATURES, f"binding lacks a signature for {s}"


def test_status_strings(lib):
    assert lib.plx_status_string(0) == b"ok"
    assert b"timed out" in lib.plx_status_string(4)
    assert lib.plx_status_string(99) == b"unknown status"


def _call_prefill(lib, fn, ptr, B=1, Hq=2, Hkv=1, L=16, d=128):
    p = ctypes.c_void_p(ptr)
    return getattr(lib, fn)(p, p, p, p, p, None, B, Hq, Hkv, L, d, None)


@pytest.mark.parametrize("fn", ["plx_prefill_fwd", "plx_prefill_fwd_f32"])
def test_prefill_rejects_bad_arguments(lib, fn):
    assert _call_prefill(lib, fn, 0) == binding.PLX_ERR_INVALID_ARG
    assert b"null" in lib.plx_last_error_message()
    assert _call_prefill(lib, fn, 4096, Hq=3, Hkv=2) == binding.PLX_ERR_INVALID_ARG
    assert b"multiple" in lib.plx_last_error_message()
    assert _call_prefill(lib, fn, 4096, L=0) == binding.PLX_ERR_INVALID_ARG
    assert _call_prefill(lib, fn, 4096, d=96) == binding.PLX_ERR_UNSUPPORTED


def test_prefill_bf16_rejects_misaligned(lib):
    assert _call_prefill(lib, "plx_prefill_fwd", 4098) == binding.PLX_ERR_INVALID_ARG
    assert b"aligned" in lib.plx_last_error_message()


def test_decode_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(4096)
    f = lib.plx_decode_fwd
    assert f(None, p, p, p, p, p, 2, 4, 2, 128, None) == binding.PLX_ERR_INVALID_ARG
    assert f(p, p, p, p, p, p, 2, 4, 2, 64, None) == binding.PLX_ERR_UNSUPPORTED
    assert f(p, p, p, p, p, p, 2, 32, 2, 128, None) == binding.PLX_ERR_UNSUPPORTED  # G = 16
    assert f(p, p, p, p, p, p, 2, 4, 3, 128, None) == binding.PLX_ERR_INVALID_ARG
    ex = lib.plx_decode_fwd_ex
    small = lib.plx_decode_workspace_bytes(2, 4, 2, 128, 3) - 4
    assert ex(p, p, p, p, p, p, 2, 4, 2, 128, 3, p, small, None) == binding.PLX_ERR_INVALID_ARG
    assert b"workspace" in lib.plx_last_error_message()


def test_workspace_size_formula(lib):
    # A row table of 8 bytes per (sequence, kv head), padded to 256 bytes, then
    # (nsplit + B * Hkv) record slots of Hq / Hkv records of 2 d + 2 floats.
    rec = (2 * 128 + 2) * 4
    assert lib.plx_decode_workspace_bytes(4, 16, 8, 128, 5) == 256 + (5 + 4 * 8) * 2 * rec
    assert lib.plx_decode_workspace_bytes(40, 4, 1, 128, 3) == 512 + (3 + 40) * 4 * rec
    assert lib.plx_decode_workspace_bytes(0, 16, 8, 128, 5) == 0
    assert lib.plx_decode_workspace_bytes(4, 16, 8, 128, 0) == 0
    assert lib.plx_decode_workspace_bytes(4, 12, 8, 128, 5) == 0  # Hq not a multiple of Hkv


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", "/nonexistent/libplx.so")
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()


def test_chunk_cor_and_train_reject_bad_arguments(lib):
    p = ctypes.c_void_p(4096)
    chunk = lib.plx_prefill_fwd_chunk
    assert chunk(p, p, p, p, p, None, 1, 2, 1, 64, 32, 128, None) == binding.PLX_ERR_INVALID_ARG
    assert b"Lk" in lib.plx_last_error_message()
    assert chunk(p, p, p, p, p, None, 1, 2, 1, 16, 64, 64, None) == binding.PLX_ERR_UNSUPPORTED
    cor = lib.plx_prefill_fwd_cor
    assert cor(p, p, p, p, p, None, None, 1, 2, 1, 16, 16, 128, None) == binding.PLX_ERR_INVALID_ARG
    assert b"cor" in lib.plx_last_error_message()
    train = lib.plx_prefill_fwd_train
    assert train(p, p, p, p, p, p, None, p, 1, 2, 1, 16, 128, None) == binding.PLX_ERR_INVALID_ARG
    assert b"o1" in lib.plx_last_error_message()
    assert train(p, p, p, p, p, p, ctypes.c_void_p(4098), p, 1, 2, 1, 16, 128,
                 None) == binding.PLX_ERR_INVALID_ARG
    assert b"aligned" in lib.plx_last_error_message()
    dcor = lib.plx_decode_fwd_cor
    assert dcor(p, p, p, p, p, p, None, 2, 4, 2, 128, None) == binding.PLX_ERR_INVALID_ARG


def test_backward_and_projection_reject_bad_arguments(lib):
    p = ctypes.c_void_p(4096)
    bwd = lib.plx_prefill_bwd
    ptrs = [p] * 13
    assert bwd(*([None] + ptrs[1:]), 1, 2, 1, 16, 128, None) == binding.PLX_ERR_INVALID_ARG
    assert bwd(*ptrs, 1, 2, 1, 16, 64, None) == binding.PLX_ERR_UNSUPPORTED
    assert bwd(*ptrs, 1, 3, 2, 16, 128, None) == binding.PLX_ERR_INVALID_ARG
    mis = ptrs[:8] + [ctypes.c_void_p(4100)] + ptrs[9:]
    assert bwd(*mis, 1, 2, 1, 16, 128, None) == binding.PLX_ERR_INVALID_ARG
    assert b"aligned" in lib.plx_last_error_message()
    proj = lib.plx_qkvr_proj
    assert proj(p, p, p, p, p, p, 1, 16, 100, 2, 1, 128, None) == binding.PLX_ERR_INVALID_ARG
    assert b"multiple of 8" in lib.plx_last_error_message()
    assert proj(p, p, p, p, p, p, 1, 16, 128, 2, 1, 64, None) == binding.PLX_ERR_UNSUPPORTED
    assert proj(p, p, None, p, p, p, 1, 16, 128, 2, 1, 128, None) == binding.PLX_ERR_INVALID_ARG


def test_noalloc_decode_rejects_bad_arguments_before_any_cuda_call(lib):
    """The allocation-free decode checks its arguments before it looks up its
    fixed array's device address: on a host without a GPU a bad call still
    gets the argument error, not a CUDA error."""
    p = ctypes.c_void_p(4096)
    f = lib.plx_decode_fwd_noalloc
    assert f(None, p, p, p, p, p, 2, 4, 2, 128, None) == binding.PLX_ERR_INVALID_ARG
    assert b"null" in lib.plx_last_error_message()
    assert f(p, p, p, p, p, p, 2, 32, 2, 128, None) == binding.PLX_ERR_UNSUPPORTED  # 16 a kv head
    assert f(p, p, p, p, p, p, 2, 4, 2, 64, None) == binding.PLX_ERR_UNSUPPORTED
    assert f(p, p, p, p, p, ctypes.c_void_p(4100), 2, 4, 2, 128, None) == binding.PLX_ERR_INVALID_ARG
    assert b"aligned" in lib.plx_last_error_message()


def test_debug_bounds_build_exports_every_symbol():
    """The PLX_DEBUG_BOUNDS build compiles for sm_103a and has the same
    interface (a CPU check; its GPU run is in test_debug_bounds_gpu.py)."""
    dbg = binding.load_debug_lib()
    for s in declared_symbols():
        assert hasattr(dbg, s), s
    assert dbg.plx_status_string(binding.PLX_ERR_BOUNDS) == b"device bounds check failed"
