"""fa_fwd_split_noalloc — the split-key forward for callers that may not
allocate device memory themselves (a plugin whose host application owns every
device allocation, or a latency-critical path that cannot take cudaMalloc's
implicit device synchronisation).  Its partial results live in a fixed array
inside the library.

Checked through the C ABI, on two calls in a row: bit-identical to
fa_fwd_split with a caller workspace (the same kernels in the same order, so
equality is exact), and against the fp64 oracle with the tolerances of the
other parity tests.  This file is collected last on purpose: if it fails, a
run that stops at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import workloads

from .parity import compare, run_oracle

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024   # FA_NOALLOC_SCRATCH_BYTES in include/fa.h


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    fa.load_library()
    yield


def _noalloc_fn():
    fn = fa.load_library().fa_fwd_split_noalloc
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


def _masked(inp, seed):
    """A key-padding mask [B, Nk] (0 / -inf) with seeded valid lengths, one of them
    shorter than a key range, so some ranges see only masked keys."""
    B, H, Nq, Nk, D = inp["shape"]
    g = torch.Generator().manual_seed(seed)
    valid = torch.randint(8, Nk + 1, (B,), generator=g)
    valid[0] = 50
    cols = torch.arange(Nk)
    m = torch.where(cols[None, :] < valid[:, None], 0.0, float("-inf")).to(torch.float32)
    inp["mask"] = m.cuda().contiguous()
    return inp


CASES = {
    # name: (workload whose value distribution is used, sizes, requested ranges)
    "d32": ("page_example", dict(B=1, H=2, Nq=256, Nk=4096), 16),
    "d64": ("sd_self", dict(B=1, H=2, Nq=300, Nk=4096), 32),
    "d128": ("hunyuan_720p", dict(B=1, H=2, Nq=256, Nk=16384), 64),
    "d64_key_mask": ("sd_cross", dict(B=2, H=2, Nq=256, Nk=1000), 8),
    "sd_cross_one_range": ("sd_cross", dict(B=2, H=8, Nq=512, Nk=80), 8),   # Nk <= 128
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_equals_workspace_entry_point_and_oracle_twice(name):
    base, sizes, splits = CASES[name]
    inp = workloads.make_inputs(base, device="cuda", **sizes)
    if name == "d64_key_mask":
        inp = _masked(inp, 7)
    B, H, Nq, Nk, D = inp["shape"]
    used = min(splits, (Nk + 127) // 128)
    if used > 1:
        assert fa.split_workspace_bytes(B, H, Nq, D, used) <= SCRATCH_BYTES
    ref_out, ref_lse = fa.fwd_split(inp["q"], inp["k"], inp["v"], mask=inp["mask"],
                                    scale=inp["scale"], num_splits=splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = run_oracle(inp)
    fn = _noalloc_fn()
    for call in range(2):
        out = torch.full_like(inp["q"], float("nan"))
        lse = torch.full((B, H, Nq), float("nan"), device="cuda")
        assert _call(fn, inp, out, lse, splits) == 0, f"call {call}"
        torch.cuda.synchronize()
        assert fa.read_device_status() == 0
        assert torch.equal(out, ref_out), f"{name} call {call}: O differs from fa_fwd_split"
        assert torch.equal(lse, ref_lse), f"{name} call {call}: LSE differs from fa_fwd_split"
        compare(out, lse, o_ref, lse_ref, label=f"noalloc {name} call {call}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fn = _noalloc_fn()
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=8, Nq=4096, Nk=2048)
    B, H, Nq, Nk, D = inp["shape"]
    assert fa.split_workspace_bytes(B, H, Nq, D, 8) > SCRATCH_BYTES
    out = torch.full_like(inp["q"], 3.0)
    lse = torch.full((B, H, Nq), 3.0, device="cuda")
    assert _call(fn, inp, out, lse, 8) == 1          # FA_ERR_INVALID_ARGUMENT, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 3.0) and torch.all(lse == 3.0)
