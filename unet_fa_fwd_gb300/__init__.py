"""GB300-native FlashAttention-style attention forward (sm_103a).

The compute lives in a C-ABI CUDA library (``csrc/``, declared in
``include/fa.h``); :mod:`unet_fa_fwd_gb300.binding` marshals torch tensors
into it.  The library is loaded on first use, and every call fails loudly if
it is missing: there is no CPU fallback.
"""
from .binding import (fa_fwd, fa_fwd_ex, fa_fwd_split, fa_fwd_status, fwd, fwd_ex,  # noqa: F401
                      fwd_split, fwd_window, window_workspace_bytes, fa_fwd_fp8, fwd_fp8,
                      fp8_workspace_bytes,
                      debug_build, debug_report, library_path, load_library, measure_ex2_rate,
                      read_device_status, split_count,
                      split_workspace_bytes, status_string, version)

__all__ = ["fa_fwd", "fa_fwd_ex", "fwd_ex", "fa_fwd_split", "fa_fwd_status", "fwd", "fwd_split", "library_path",
           "load_library", "read_device_status", "split_count", "split_workspace_bytes",
           "debug_build", "debug_report",
           "status_string", "version", "fwd_window", "window_workspace_bytes", "fa_fwd_fp8",
           "fwd_fp8", "fp8_workspace_bytes", "measure_ex2_rate"]
