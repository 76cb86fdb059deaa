"""Python binding of the C ABI in ``include/fa.h`` (argument marshalling only).

Torch provides device memory and streams; every step of the attention forward
runs in the CUDA library.  The library is loaded on first use; if it is
missing or cannot be loaded every call raises — there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import _build

FA_OK = 0
FA_ERR_INVALID_ARGUMENT = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_DEBUG_CHECK = 5

FA_MASK_NONE = 0
FA_MASK_KEY_PADDING = 1
FA_MASK_ADDITIVE = 2
FA_MASK_BOOL = 3

_lib = None
_lock = threading.Lock()


class FaMask(ctypes.Structure):
    """The C struct fa_mask."""
    _fields_ = [("kind", ctypes.c_int), ("data", ctypes.c_void_p), ("heads", ctypes.c_int)]


def library_path() -> str:
    """The release library, or with FA_DEBUG=1 in the environment the debug build
    (device-side bounds and schedule checks; see fa_debug_report)."""
    return _build.LIB_DEBUG if os.environ.get("FA_DEBUG") == "1" else _build.LIB


def load_library() -> ctypes.CDLL:
    """Load ``libfa_fwd.so`` (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: build it first (python -c 'import "
                    "__graft_entry__ as g; g.build()'); there is no CPU fallback")
            lib = ctypes.CDLL(path)
            vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
            lib.fa_fwd.restype = i32
            lib.fa_fwd_ex.argtypes = [vp, vp, vp, ctypes.POINTER(FaMask), i32, vp, vp, i32, i32, i32,
                                      i32, i32, f32, vp]
            lib.fa_fwd_ex.restype = i32
            sz = ctypes.c_size_t
            lib.fa_fwd_window.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                          i32, f32, vp, sz, vp]
            lib.fa_fwd_window.restype = i32
            lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, sz, vp]
            lib.fa_fwd_fp8.restype = i32
            lib.fa_fp8_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            lib.fa_fp8_workspace_bytes.restype = sz
            lib.fa_window_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            lib.fa_window_workspace_bytes.restype = sz
            lib.fa_fwd_split.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32,
                                         vp, sz, vp]
            lib.fa_fwd_split.restype = i32
            lib.fa_split_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            lib.fa_split_workspace_bytes.restype = sz
            lib.fa_split_count.argtypes = [i32, i32, i32, i32, i32]
            lib.fa_split_count.restype = i32
            lib.fa_read_device_status.argtypes = [vp, ctypes.POINTER(i32)]
            lib.fa_read_device_status.restype = i32
            lib.fa_measure_ex2_rate.argtypes = [vp, ctypes.POINTER(ctypes.c_double)]
            lib.fa_measure_ex2_rate.restype = i32
            lib.fa_status_string.argtypes = [i32]
            lib.fa_status_string.restype = ctypes.c_char_p
            lib.fa_version.argtypes = []
            lib.fa_version.restype = ctypes.c_char_p
            lib.fa_debug_build.argtypes = []
            lib.fa_debug_build.restype = i32
            lib.fa_debug_report.argtypes = [vp, ctypes.POINTER(i32)]
            lib.fa_debug_report.restype = i32
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load_library().fa_status_string(int(code)).decode()


def version() -> str:
    return load_library().fa_version().decode()


def _stream_handle(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def fa_fwd_status(q_ptr: int, k_ptr: int, v_ptr: int, mask_ptr: int | None, out_ptr: int,
                  lse_ptr: int, B: int, H: int, Nq: int, Nk: int, D: int, scale: float,
                  stream: int | None) -> int:
    """Raw call with integer pointers; returns the status code."""
    return load_library().fa_fwd(q_ptr, k_ptr, v_ptr, mask_ptr, out_ptr, lse_ptr, B, H, Nq, Nk, D,
                                 ctypes.c_float(scale), stream)


def _check(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor | None,
           out: torch.Tensor, lse: torch.Tensor, scale: float | None = None, stream=None) -> None:
    """Enqueue the forward into caller-provided ``out`` (bf16 [B,H,Nq,D]) and ``lse`` (fp32 [B,H,Nq])."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, D]")
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    _check(q, "q", torch.bfloat16, (B, H, Nq, D))
    _check(k, "k", torch.bfloat16, (B, H, Nk, D))
    _check(v, "v", torch.bfloat16, (B, H, Nk, D))
    _check(out, "out", torch.bfloat16, (B, H, Nq, D))
    _check(lse, "lse", torch.float32, (B, H, Nq))
    if mask is not None:
        _check(mask, "mask", torch.float32, (B, Nk))
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = fa_fwd_status(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                       None if mask is None else mask.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, H, Nq, Nk, D, float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise RuntimeError(f"fa_fwd failed: {status_string(rc)}")


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor | None = None,
        scale: float | None = None, stream=None):
    """Allocate outputs and run the forward; returns (O bf16 [B,H,Nq,D], LSE fp32 [B,H,Nq])."""
    B, H, Nq, D = q.shape
    out = torch.empty((B, H, Nq, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, mask, out, lse, scale=scale, stream=stream)
    return out, lse


def fa_fwd_ex(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
              lse: torch.Tensor, key_mask: torch.Tensor | None = None,
              full_mask: torch.Tensor | None = None, causal: bool = False,
              scale: float | None = None, stream=None) -> None:
    """Forward with general masks into caller buffers.

    key_mask: fp32 [B, Nk] additive; full_mask: fp32 [B, 1|H, Nq, Nk] additive or
    bool/uint8 [B, 1|H, Nq, Nk] (True/nonzero keeps the pair); causal: exclude key j > query i.
    At most one of key_mask / full_mask.
    """
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    _check(q, "q", torch.bfloat16, (B, H, Nq, D))
    _check(k, "k", torch.bfloat16, (B, H, Nk, D))
    _check(v, "v", torch.bfloat16, (B, H, Nk, D))
    _check(out, "out", torch.bfloat16, (B, H, Nq, D))
    _check(lse, "lse", torch.float32, (B, H, Nq))
    if key_mask is not None and full_mask is not None:
        raise ValueError("pass key_mask or full_mask, not both")
    m = FaMask(FA_MASK_NONE, None, 1)
    if key_mask is not None:
        _check(key_mask, "key_mask", torch.float32, (B, Nk))
        m = FaMask(FA_MASK_KEY_PADDING, key_mask.data_ptr(), 1)
    elif full_mask is not None:
        if full_mask.dim() != 4 or full_mask.shape[1] not in (1, H):
            raise ValueError("full_mask must be [B, 1|H, Nq, Nk]")
        heads = full_mask.shape[1]
        if full_mask.dtype == torch.float32:
            _check(full_mask, "full_mask", torch.float32, (B, heads, Nq, Nk))
            m = FaMask(FA_MASK_ADDITIVE, full_mask.data_ptr(), heads)
        elif full_mask.dtype in (torch.bool, torch.uint8):
            _check(full_mask, "full_mask", full_mask.dtype, (B, heads, Nq, Nk))
            m = FaMask(FA_MASK_BOOL, full_mask.data_ptr(), heads)
        else:
            raise TypeError("full_mask must be float32 (additive) or bool/uint8")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = load_library().fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(m),
                                   int(bool(causal)), out.data_ptr(), lse.data_ptr(), B, H, Nq, Nk,
                                   D, ctypes.c_float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise RuntimeError(f"fa_fwd_ex failed: {status_string(rc)}")


def fwd_ex(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, key_mask: torch.Tensor | None = None,
           full_mask: torch.Tensor | None = None, causal: bool = False,
           scale: float | None = None, stream=None):
    """Allocate outputs and run fa_fwd_ex; returns (O, LSE)."""
    B, H, Nq, D = q.shape
    out = torch.empty((B, H, Nq, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    fa_fwd_ex(q, k, v, out, lse, key_mask=key_mask, full_mask=full_mask, causal=causal,
              scale=scale, stream=stream)
    return out, lse


def fp8_workspace_bytes(B: int, H: int, Nq: int, Nk: int, D: int) -> int:
    return int(load_library().fa_fp8_workspace_bytes(B, H, Nq, Nk, D))


def fa_fwd_fp8(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor | None,
               out: torch.Tensor, lse: torch.Tensor, workspace: torch.Tensor,
               scale: float | None = None, stream=None) -> None:
    """FP8 (e4m3) Q K^T forward into caller buffers; `workspace` holds at least
    fp8_workspace_bytes(...) bytes."""
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    _check(q, "q", torch.bfloat16, (B, H, Nq, D))
    _check(k, "k", torch.bfloat16, (B, H, Nk, D))
    _check(v, "v", torch.bfloat16, (B, H, Nk, D))
    _check(out, "out", torch.bfloat16, (B, H, Nq, D))
    _check(lse, "lse", torch.float32, (B, H, Nq))
    if mask is not None:
        _check(mask, "mask", torch.float32, (B, Nk))
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = load_library().fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                    None if mask is None else mask.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), B, H, Nq, Nk, D, ctypes.c_float(scale),
                                    workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                    _stream_handle(stream))
    if rc != FA_OK:
        raise RuntimeError(f"fa_fwd_fp8 failed: {status_string(rc)}")


def fwd_fp8(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor | None = None,
            scale: float | None = None, stream=None):
    """Allocate outputs and workspace (torch) and run the FP8 Q K^T forward."""
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    out = torch.empty((B, H, Nq, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    ws = torch.empty(fp8_workspace_bytes(B, H, Nq, Nk, D), dtype=torch.uint8, device=q.device)
    fa_fwd_fp8(q, k, v, mask, out, lse, ws, scale=scale, stream=stream)
    return out, lse


def window_workspace_bytes(B: int, H: int, img_h: int, img_w: int, D: int) -> int:
    return int(load_library().fa_window_workspace_bytes(B, H, img_h, img_w, D))


def fwd_window(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, img_h: int, img_w: int,
               win_h: int, win_w: int, shift_h: int = 0, shift_w: int = 0,
               scale: float | None = None, stream=None):
    """Window / shifted-window attention; q, k, v bf16 [B, H, img_h*img_w, D] in grid order.
    Allocates the outputs with torch (no workspace is needed); returns (O, LSE)."""
    B, H, N, D = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, (B, H, N, D))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    ws_bytes = window_workspace_bytes(B, H, img_h, img_w, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = load_library().fa_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       lse.data_ptr(), B, H, img_h, img_w, D, win_h, win_w,
                                       shift_h, shift_w, ctypes.c_float(scale),
                                       None if ws is None else ws.data_ptr(), ws_bytes,
                                       _stream_handle(stream))
    if rc != FA_OK:
        raise RuntimeError(f"fa_fwd_window failed: {status_string(rc)}")
    return out, lse


def split_workspace_bytes(B: int, H: int, Nq: int, D: int, num_splits: int) -> int:
    return int(load_library().fa_split_workspace_bytes(B, H, Nq, D, num_splits))


def split_count(B: int, H: int, Nq: int, Nk: int, num_sms: int | None = None) -> int:
    """Key-range count the library recommends for these sizes on this GPU."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return int(load_library().fa_split_count(B, H, Nq, Nk, num_sms))


def fa_fwd_split(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor | None,
                 out: torch.Tensor, lse: torch.Tensor, num_splits: int,
                 workspace: torch.Tensor | None, scale: float | None = None, stream=None) -> None:
    """Split-key forward into caller buffers; `workspace` is a device tensor of at least
    split_workspace_bytes(...) bytes (any dtype, contiguous), or None for one range."""
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    _check(q, "q", torch.bfloat16, (B, H, Nq, D))
    _check(k, "k", torch.bfloat16, (B, H, Nk, D))
    _check(v, "v", torch.bfloat16, (B, H, Nk, D))
    _check(out, "out", torch.bfloat16, (B, H, Nq, D))
    _check(lse, "lse", torch.float32, (B, H, Nq))
    if mask is not None:
        _check(mask, "mask", torch.float32, (B, Nk))
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = load_library().fa_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                      None if mask is None else mask.data_ptr(), out.data_ptr(),
                                      lse.data_ptr(), B, H, Nq, Nk, D, ctypes.c_float(scale),
                                      int(num_splits), ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != FA_OK:
        raise RuntimeError(f"fa_fwd_split failed: {status_string(rc)}")


def fwd_split(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor | None = None,
              scale: float | None = None, num_splits: int | None = None, stream=None):
    """Allocate outputs and workspace (torch) and run the split-key forward."""
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if num_splits is None:
        num_splits = split_count(B, H, Nq, Nk)
    out = torch.empty((B, H, Nq, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    ws = torch.empty(split_workspace_bytes(B, H, Nq, D, num_splits), dtype=torch.uint8,
                     device=q.device)
    fa_fwd_split(q, k, v, mask, out, lse, num_splits, ws, scale=scale, stream=stream)
    return out, lse


def measure_ex2_rate(stream=None) -> float:
    """Exponentials (ex2.approx.ftz.f32) one SM completes per SM clock, measured on the device."""
    rate = ctypes.c_double(0.0)
    rc = load_library().fa_measure_ex2_rate(_stream_handle(stream), ctypes.byref(rate))
    if rc != FA_OK:
        raise RuntimeError(f"fa_measure_ex2_rate failed: {status_string(rc)}")
    return rate.value


def read_device_status(stream=None) -> int:
    """Synchronise and return (then reset) the device status word: FA_OK or FA_ERR_TIMEOUT."""
    st = ctypes.c_int(0)
    rc = load_library().fa_read_device_status(_stream_handle(stream), ctypes.byref(st))
    if rc != FA_OK:
        raise RuntimeError(f"fa_read_device_status failed: {status_string(rc)}")
    return st.value


def debug_build() -> bool:
    """True when the loaded library is the debug build."""
    return bool(load_library().fa_debug_build())


def debug_report(stream=None) -> list[int]:
    """Synchronise and return (then clear) the first failed device-side check of a
    debug build: [check id, CTA, thread, a, b, 0, 0, failures]; all zeros if none."""
    rec = (ctypes.c_int * 8)()
    rc = load_library().fa_debug_report(_stream_handle(stream), rec)
    if rc != FA_OK:
        raise RuntimeError(f"fa_debug_report failed: {status_string(rc)}")
    return list(rec)
