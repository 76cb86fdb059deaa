"""fa_fwd_split_noalloc — the split-key forward for callers that may not
allocate device memory themselves (its scratch is a fixed array inside the
library).  Checked through the C ABI against fa_fwd_split with a caller
workspace, on two calls in a row, with the tolerances of the other parity
tests.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

import unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import workloads

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024   # FA_NOALLOC_SCRATCH_BYTES in include/fa.h


def _noalloc_fn():
    lib = fa.load_library()
    fn = lib.fa_fwd_split_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32, vp]
    fn.restype = i32
    return fn


def _call(fn, inp, out, lse, splits):
    B, H, Nq, Nk, D = inp["shape"]
    mask = inp["mask"]
    return fn(inp["q"].data_ptr(), inp["k"].data_ptr(), inp["v"].data_ptr(),
              None if mask is None else mask.data_ptr(), out.data_ptr(), lse.data_ptr(),
              B, H, Nq, Nk, D, inp["scale"], splits, torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_twice():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    fn = _noalloc_fn()
    inp = workloads.make_inputs("hunyuan_720p", device="cuda", B=1, H=2, Nq=256, Nk=16384)
    B, H, Nq, Nk, D = inp["shape"]
    splits = 64
    assert fa.split_workspace_bytes(B, H, Nq, D, splits) <= SCRATCH_BYTES
    ref_out, ref_lse = fa.fwd_split(inp["q"], inp["k"], inp["v"], scale=inp["scale"],
                                    num_splits=splits)
    for call in range(2):
        out = torch.full_like(inp["q"], float("nan"))
        lse = torch.full((B, H, Nq), float("nan"), device="cuda")
        assert _call(fn, inp, out, lse, splits) == 0
        torch.cuda.synchronize()
        assert fa.read_device_status() == 0
        err = (out.float() - ref_out.float()).abs()
        assert torch.isfinite(out.float()).all(), f"call {call}"
        assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3, f"call {call}"
        lrel = (lse - ref_lse).abs() / ref_lse.abs().clamp_min(1.0)
        assert lrel.max().item() <= 1e-3, f"call {call}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    torch.cuda.set_device(0)
    fn = _noalloc_fn()
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=8, Nq=4096, Nk=2048)
    B, H, Nq, Nk, D = inp["shape"]
    assert fa.split_workspace_bytes(B, H, Nq, D, 8) > SCRATCH_BYTES
    out = torch.full_like(inp["q"], 3.0)
    lse = torch.full((B, H, Nq), 3.0, device="cuda")
    assert _call(fn, inp, out, lse, 8) == 1          # FA_ERR_INVALID_ARGUMENT, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 3.0) and torch.all(lse == 3.0)
