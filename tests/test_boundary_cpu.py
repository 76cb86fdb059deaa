"""The C-ABI library loads on a machine without a GPU, exports every function
include/fa.h declares, and validates arguments before any CUDA call."""
import ctypes
import os
import re

import pytest
import torch

import unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(fa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.load_library()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"fa_fwd", "fa_status_string", "fa_version", "fa_read_device_status",
            "fa_measure_ex2_rate"} <= set(names)
    raw = ctypes.CDLL(_build.LIB)
    for n in names:
        assert hasattr(raw, n), n


def test_debug_library_exports_the_same_symbols(lib):
    """The debug build (device-side checks) exports every declared function too,
    and each library reports which build it is."""
    names = _declared()
    dbg = ctypes.CDLL(_build.LIB_DEBUG)
    for n in names:
        assert hasattr(dbg, n), n
    rel = ctypes.CDLL(_build.LIB)
    assert rel.fa_debug_build() == 0 and dbg.fa_debug_build() == 1
    assert dbg.fa_debug_report(None, None) == 1     # FA_ERR_INVALID_ARGUMENT, no CUDA call


def test_strings(lib):
    assert fa.version().startswith("unet_fa_fwd_gb300")
    assert fa.status_string(0) == "FA_OK"
    assert fa.status_string(4) == "FA_ERR_TIMEOUT"
    assert fa.status_string(5) == "FA_ERR_DEBUG_CHECK"
    assert fa.status_string(99) == "FA_ERR_UNKNOWN"


FAKE = dict(q=0x10000, k=0x20000, v=0x30000, mask=None, out=0x40000, lse=0x50000,
            B=1, H=2, Nq=100, Nk=100, D=64, scale=0.125, stream=None)


def _call(**kw):
    a = dict(FAKE, **kw)
    return fa.fa_fwd_status(a["q"], a["k"], a["v"], a["mask"], a["out"], a["lse"], a["B"], a["H"],
                            a["Nq"], a["Nk"], a["D"], a["scale"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(out=None), 1),
    (dict(lse=None), 1), (dict(B=0), 1), (dict(H=-1), 1), (dict(Nq=0), 1), (dict(Nk=0), 1),
    (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1),
    (dict(D=48), 2), (dict(D=256), 2), (dict(D=16), 2),
    (dict(q=0x10008), 1), (dict(lse=0x50004), 1), (dict(mask=0x60004), 1),
    (dict(out=0x10000), 1),                  # out aliases q
    (dict(lse=0x40000 + 64), 1),             # lse inside out
    (dict(mask=0x40000 + 32), 1),            # mask inside out
    (dict(B=1 << 20, H=1 << 12), 1),         # B*H overflows int32
])
def test_validation_before_any_cuda_call(lib, kw, code):
    assert _call(**kw) == code


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call() == 3


def test_fault_injection_hook(lib, monkeypatch):
    monkeypatch.setenv("FA_FAULT_INJECT", "launch")
    assert _call() == 3


def test_split_workspace_and_count(lib):
    assert fa.split_workspace_bytes(1, 24, 256, 128, 4) == (
        ((24 * 256 * 4 * 128 * 4 + 255) // 256) * 256 + ((24 * 256 * 4 * 4 + 255) // 256) * 256)
    assert fa.split_workspace_bytes(0, 1, 1, 64, 1) == 0
    assert fa.split_workspace_bytes(1, 1, 1, 64, 0) == 0
    # enough units already: no split
    assert fa.split_count(1, 24, 16896, 16896, num_sms=152) == 1
    # one head, 256 queries, 119056 keys (931 key blocks): fill 152 SMs
    assert fa.split_count(1, 1, 256, 119056, num_sms=152) == 152
    # short key set: at least four key blocks per range
    assert fa.split_count(1, 1, 128, 1024, num_sms=152) == 2
    assert fa.split_count(1, 1, 128, 100, num_sms=152) == 1


def _split_call(**kw):
    a = dict(FAKE, num_splits=4, ws=0x80000, ws_bytes=1 << 30)
    a.update(kw)
    return fa.load_library().fa_fwd_split(a["q"], a["k"], a["v"], a["mask"], a["out"], a["lse"],
                                          a["B"], a["H"], a["Nq"], 1000, a["D"],
                                          ctypes.c_float(a["scale"]), a["num_splits"], a["ws"],
                                          a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(num_splits=0), 1), (dict(ws=None), 1), (dict(ws=0x80008), 1), (dict(ws_bytes=1024), 1),
    (dict(D=48), 2), (dict(q=None), 1),
])
def test_split_validation_before_any_cuda_call(lib, kw, code):
    assert _split_call(**kw) == code


def test_fa_fwd_ex_mask_validation_before_any_cuda_call(lib):
    from unet_fa_fwd_gb300.binding import FaMask
    raw = fa.load_library()
    a = FAKE
    for kind, data, heads, code in [(7, 0x1000, 1, 1), (2, None, 1, 1), (2, 0x1002, 1, 1),
                                    (3, 0x1000, 5, 1), (1, None, 1, 1)]:
        m = FaMask(kind, data, heads)
        rc = raw.fa_fwd_ex(a["q"], a["k"], a["v"], ctypes.byref(m), 0, a["out"], a["lse"], a["B"],
                           a["H"], a["Nq"], a["Nk"], a["D"], ctypes.c_float(a["scale"]), None)
        assert rc == code, (kind, data, heads)
    # a valid call without a GPU reaches the CUDA set-up and fails there
    import torch
    if not torch.cuda.is_available():
        m = FaMask(3, 0x90000, 2)
        rc = raw.fa_fwd_ex(a["q"], a["k"], a["v"], ctypes.byref(m), 1, a["out"], a["lse"], a["B"],
                           a["H"], a["Nq"], a["Nk"], a["D"], ctypes.c_float(a["scale"]), None)
        assert rc == 3


def test_window_validation_before_any_cuda_call(lib):
    raw = fa.load_library()
    # the attention kernel gathers and scatters window rows itself: no workspace
    assert fa.window_workspace_bytes(1, 2, 8, 8, 64) == 0
    assert fa.window_workspace_bytes(0, 2, 8, 8, 64) == 0

    def call(img=(8, 8), win=(4, 4), D=64, ws=None, ws_bytes=0, q=0x10000, B=1, out=0x40000):
        return raw.fa_fwd_window(q, 0x20000, 0x30000, out, 0x50000, B, 2, img[0], img[1], D,
                                 win[0], win[1], 1, 1, ctypes.c_float(0.1), ws, ws_bytes, None)
    assert call(win=(3, 4)) == 1       # windows must tile the grid
    assert call(win=(0, 4)) == 1
    assert call(D=48) == 2
    assert call(q=None) == 1
    assert call(q=0x10008) == 1        # misaligned tensor
    assert call(out=0x10000) == 1      # O overlaps Q
    assert call(B=1 << 20, img=(64, 64), win=(8, 8)) == 1   # 2^31 rows or more
    if not torch.cuda.is_available():
        # valid arguments (any workspace): the first CUDA call fails on this machine
        assert call() == 3 and call(ws=0xA0000, ws_bytes=1 << 20) == 3


def test_fp8_validation_before_any_cuda_call(lib):
    raw = fa.load_library()
    need = fa.fp8_workspace_bytes(1, 2, 100, 100, 64)
    assert need > 2 * 100 * 64 * 2 and fa.fp8_workspace_bytes(1, 2, 100, 100, 48) == 0

    def call(ws=0xA0000, ws_bytes=1 << 24, D=64, q=0x10000):
        return raw.fa_fwd_fp8(q, 0x20000, 0x30000, None, 0x40000, 0x50000, 1, 2, 100, 100, D,
                              ctypes.c_float(0.1), ws, ws_bytes, None)
    assert call(ws=None) == 1
    assert call(ws=0xA0008) == 1
    assert call(ws_bytes=need - 1) == 1
    assert call(D=48) == 2
    assert call(q=None) == 1


def test_ex2_probe_validation_before_any_cuda_call(lib):
    assert lib.fa_measure_ex2_rate(None, None) == 1   # FA_ERR_INVALID_ARGUMENT


def _noalloc_call(**kw):
    a = dict(FAKE, num_splits=4)
    a.update(kw)
    fn = fa.load_library().fa_fwd_split_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32, vp]
    fn.restype = i32
    return fn(a["q"], a["k"], a["v"], a["mask"], a["out"], a["lse"], a["B"], a["H"], a["Nq"],
              a["Nk"], a["D"], a["scale"], a["num_splits"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(num_splits=0), 1), (dict(num_splits=-3), 1), (dict(Nk=0), 1), (dict(B=0), 1),
    (dict(Nq=0), 1), (dict(q=None), 1), (dict(q=None, Nk=1000), 1), (dict(lse=None), 1),
    (dict(out=0x10000), 1), (dict(scale=float("nan")), 1), (dict(D=48), 2),
    (dict(D=48, Nk=1000), 2),
    # 8 heads x 4096 queries x 8 ranges of fp32 partials do not fit the 32 MiB scratch
    (dict(B=1, H=8, Nq=4096, Nk=2048, D=128, num_splits=8, q=1 << 40, k=2 << 40, v=3 << 40,
          out=4 << 40, lse=5 << 40), 1),
])
def test_noalloc_validation_before_any_cuda_call(lib, kw, code):
    """Every rejection of fa_fwd_split_noalloc happens before its first CUDA call
    (on this machine without a driver a CUDA call would answer FA_ERR_CUDA)."""
    assert _noalloc_call(**kw) == code


def test_noalloc_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _noalloc_call(Nk=100, num_splits=1) == 3     # one range: the plain forward's set-up
    far = dict(q=1 << 40, k=2 << 40, v=3 << 40, out=4 << 40, lse=5 << 40)
    assert _noalloc_call(Nk=1000, num_splits=4, **far) == 3    # scratch look-up


def test_split_unit_count_overflow_rejected_before_any_cuda_call(lib):
    # B*H = 2^24 heads x 1 query pair x 256 key ranges = 2^32 work units > INT_MAX.
    ptrs = dict(q=1 << 47, k=2 << 47, v=3 << 47, out=4 << 47, lse=5 << 47)
    raw = fa.load_library()
    rc = raw.fa_fwd_split(ptrs["q"], ptrs["k"], ptrs["v"], None, ptrs["out"], ptrs["lse"],
                          1 << 14, 1 << 10, 256, 256 * 128, 64, ctypes.c_float(0.125), 256,
                          1 << 52, 1 << 60, None)
    assert rc == 1


def test_window_fault_hook_enqueues_nothing(lib, monkeypatch):
    """With valid arguments the window path sets up (where the launch hook fires)
    before its first kernel is enqueued."""
    monkeypatch.setenv("FA_FAULT_INJECT", "launch")
    raw = fa.load_library()
    rc = raw.fa_fwd_window(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 1, 2, 8, 8, 64, 4, 4, 0, 0,
                           ctypes.c_float(0.1), 0xA0000, 1 << 20, None)
    assert rc == 3
