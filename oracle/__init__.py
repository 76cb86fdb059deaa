"""CPU oracle for the non-causal attention forward — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The product path (the CUDA library
and its Python binding) never does.

The arithmetic lives in ``fa_oracle.c`` (plain C, fp64): it materialises each
score row, applies scale then the additive key mask, takes a two-pass softmax
and the weighted sum of V, and the natural-log row LSE.  This module only
marshals numpy arrays into that library with ``ctypes``.

Sources: "算子加速：注意力、编译与融合" (anrans.github.io, perf/kernels), section
"注意力：从O(N²)显存到分块", function ``naive``; "FlashAttention原理与工业实战"
§2.1 (masked keys become -inf) and §2.3 (the kernel writes a row Lse);
"Step 3.7 Flash" §2.3 (scale first, then add the mask).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

DTYPE_F32 = 0
DTYPE_BF16 = 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        vp, dp, i32, f64 = ctypes.c_void_p, ctypes.POINTER(ctypes.c_double), ctypes.c_int, ctypes.c_double
        lib.fa_oracle_fwd.argtypes = [vp, vp, vp, vp, i32, dp, dp, i32, i32, i32, i32, i32, f64, i32]
        lib.fa_oracle_fwd.restype = i32
        lib.fa_oracle_rows.argtypes = [vp, vp, vp, vp, i32, vp, i32, dp, dp, i32, i32, i32, i32, i32,
                                       f64, i32]
        lib.fa_oracle_rows.restype = i32
        lib.fa_oracle_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp, i32, dp, dp, i32,
                                         i32, i32, i32, i32, f64, i32]
        lib.fa_oracle_fwd_ex.restype = i32
        lib.fa_oracle_window.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, dp, dp, i32,
                                         i32, i32, f64, i32]
        lib.fa_oracle_window.restype = i32
        lib.fa_oracle_probs.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, dp, dp, dp, i32, i32,
                                        i32, i32, i32, f64]
        lib.fa_oracle_probs.restype = i32
        _lib = lib
    return _lib


def default_threads() -> int:
    return os.cpu_count() or 1


def _as_input(x: np.ndarray):
    """Return (contiguous array, dtype code).  uint16/int16 arrays are raw bf16 bits."""
    if x.dtype in (np.uint16, np.int16):
        return np.ascontiguousarray(x).view(np.uint16), DTYPE_BF16
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), DTYPE_F32
    if x.dtype == np.float64:
        # fp64 inputs are accepted only when they are exactly fp32 values.
        x32 = x.astype(np.float32)
        if not np.array_equal(x32.astype(np.float64), x, equal_nan=True):
            raise ValueError("fp64 oracle input is not exactly representable in fp32")
        return np.ascontiguousarray(x32), DTYPE_F32
    raise TypeError(f"unsupported oracle input dtype {x.dtype}")


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray | None = None,
              scale: float | None = None, rows: np.ndarray | None = None,
              nthreads: int | None = None):
    """fp64 attention forward.

    q: [B,H,Nq,D]; k, v: [B,H,Nk,D] — fp32, or uint16 raw bf16 bits (all the same kind).
    mask: optional fp32 [B,Nk] additive key mask (-inf = ignore).
    scale: multiplies q.k (default 1/sqrt(D)).
    rows: optional int64 [B*H, nrows] query indices per head (sampled mode).
    Returns (O, LSE): fp64 [B,H,Nq|nrows,D] and [B,H,Nq|nrows].
    """
    lib = _load()
    B, H, Nq, D = q.shape
    Bk, Hk, Nk, Dk = k.shape
    if (Bk, Hk, Dk) != (B, H, D) or v.shape != k.shape:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    qa, dt = _as_input(q)
    ka, dtk = _as_input(k)
    va, dtv = _as_input(v)
    if not (dt == dtk == dtv):
        raise TypeError("q, k, v must share one dtype")
    m = None
    if mask is not None:
        m = np.ascontiguousarray(mask, dtype=np.float32)
        if m.shape != (B, Nk):
            raise ValueError(f"mask must be [B,Nk]=({B},{Nk}), got {m.shape}")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    nthreads = nthreads or default_threads()
    if rows is None:
        out = np.empty((B, H, Nq, D), dtype=np.float64)
        lse = np.empty((B, H, Nq), dtype=np.float64)
        rc = lib.fa_oracle_fwd(_ptr(qa), _ptr(ka), _ptr(va), _ptr(m), dt,
                               out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                               lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                               B, H, Nq, Nk, D, float(scale), int(nthreads))
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        if r.ndim != 2 or r.shape[0] != B * H:
            raise ValueError("rows must be [B*H, nrows]")
        nrows = r.shape[1]
        out = np.empty((B, H, nrows, D), dtype=np.float64)
        lse = np.empty((B, H, nrows), dtype=np.float64)
        rc = lib.fa_oracle_rows(_ptr(qa), _ptr(ka), _ptr(va), _ptr(m), dt, _ptr(r), nrows,
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                B, H, Nq, Nk, D, float(scale), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return out, lse


def attention_ex(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray | None = None,
                 full_mask: np.ndarray | None = None, causal: bool = False,
                 scale: float | None = None, rows: np.ndarray | None = None,
                 nthreads: int | None = None):
    """fp64 forward with general masking.

    mask: key-padding fp32 [B,Nk]; full_mask: additive fp32 [B, 1|H, Nq, Nk];
    causal: exclude key j > query i.  Other arguments as attention().
    """
    lib = _load()
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    qa, dt = _as_input(q)
    ka, _ = _as_input(k)
    va, _ = _as_input(v)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.float32)
    fm, mh = None, 1
    if full_mask is not None:
        fm = np.ascontiguousarray(full_mask, dtype=np.float32)
        if fm.ndim != 4 or fm.shape[0] != B or fm.shape[2:] != (Nq, Nk) or fm.shape[1] not in (1, H):
            raise ValueError(f"full_mask must be [B, 1|H, Nq, Nk], got {fm.shape}")
        mh = fm.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    r, nrows = None, Nq
    if rows is not None:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = r.shape[1]
    out = np.empty((B, H, nrows, D), dtype=np.float64)
    lse = np.empty((B, H, nrows), dtype=np.float64)
    rc = lib.fa_oracle_fwd_ex(_ptr(qa), _ptr(ka), _ptr(va), _ptr(m), _ptr(fm), mh, int(bool(causal)),
                              dt, _ptr(r), nrows if r is not None else 0,
                              out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                              lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                              B, H, Nq, Nk, D, float(scale), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return out, lse


def window_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, img_h: int, img_w: int,
                     win_h: int, win_w: int, shift_h: int = 0, shift_w: int = 0,
                     scale: float | None = None, nthreads: int | None = None):
    """fp64 window / shifted-window attention on an img_h x img_w token grid.

    q, k, v: [B, H, img_h*img_w, D] in row-major token order.  Returns (O, LSE)
    in the same order.
    """
    lib = _load()
    B, H, N, D = q.shape
    if N != img_h * img_w or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must be [B, H, img_h*img_w, D]")
    qa, dt = _as_input(q)
    ka, _ = _as_input(k)
    va, _ = _as_input(v)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.empty((B, H, N, D), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = lib.fa_oracle_window(_ptr(qa), _ptr(ka), _ptr(va), dt, img_h, img_w, win_h, win_w,
                              shift_h, shift_w,
                              out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                              lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                              B, H, D, float(scale), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return out, lse


def probs(q: np.ndarray, k: np.ndarray, v: np.ndarray, b: int, h: int, i: int,
          mask: np.ndarray | None = None, scale: float | None = None):
    """Row (b, h, i) through the oracle's own row function: returns (p, o_row, lse) with
    p the softmax row p_ij (fp64, length Nk), o_row the O row (fp64, length D)."""
    lib = _load()
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    qa, dt = _as_input(q)
    ka, dtk = _as_input(k)
    va, dtv = _as_input(v)
    if not (dt == dtk == dtv):
        raise TypeError("q, k, v must share one dtype")
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.float32)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dp = ctypes.POINTER(ctypes.c_double)
    p = np.empty(Nk, dtype=np.float64)
    o_row = np.empty(D, dtype=np.float64)
    lse = ctypes.c_double(0.0)
    rc = lib.fa_oracle_probs(_ptr(qa), _ptr(ka), _ptr(va), _ptr(m), dt, b, h, i,
                             p.ctypes.data_as(dp), o_row.ctypes.data_as(dp), ctypes.byref(lse),
                             B, H, Nq, Nk, D, float(scale))
    if rc != 0:
        raise RuntimeError(f"oracle probs failed with code {rc}")
    return p, o_row, lse.value
