"""GB300-native Parallax (parametrized local linear attention) forward.

The compute lives in libplx.so (C ABI in include/plx.h, kernels in csrc/);
``binding`` exposes each entry point under its C name. ``inputs`` draws the
seeded synthetic workloads. Importing this package does not load the library;
the first call does, and raises if it has not been built.
"""
from .binding import (PlxError, plx_check_device_error, plx_debug_timeout_probe,  # noqa: F401
                      plx_decode_default_nsplit, plx_decode_fwd, plx_decode_fwd_cor,
                      plx_decode_fwd_noalloc, plx_decode_workspace_bytes,
                      plx_prefill_bwd, plx_prefill_fwd, plx_prefill_fwd_chunk,
                      plx_prefill_fwd_cor, plx_prefill_fwd_f32, plx_prefill_fwd_train,
                      plx_qkvr_proj)
