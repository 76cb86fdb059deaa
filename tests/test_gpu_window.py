"""GPU parity of fa_fwd_window (window / shifted-window attention: gather,
attention, scatter) against the oracle's fa_oracle_window."""
import pytest
import torch

import oracle
import unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import workloads

from .parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.load_library()
    torch.cuda.set_device(0)
    yield


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("img,win,shift", [
    ((16, 16), (8, 8), (0, 0)),
    ((16, 16), (8, 8), (4, 4)),          # Swin-style half-window shift
    ((14, 21), (7, 7), (3, 3)),          # 7x7 windows, non-square grid
    ((32, 16), (16, 8), (5, 2)),         # 128-token windows
    ((12, 12), (12, 12), (0, 0)),        # one window = full attention
    ((16, 16), (4, 4), (2, 2)),          # 16-token windows: 8 per 128-row batch entry
    ((8, 8), (2, 2), (1, 1)),            # 4-token windows: 32 per entry
    ((12, 8), (4, 4), (0, 0)),           # 12 windows in all: packing falls back to 6 per entry
    ((32, 32), (8, 8), (3, 5)),          # 16 windows of 64 per image, 4 per entry, odd shifts
])
def test_window_parity(D, img, win, shift):
    base = {32: "page_example", 64: "sd_self", 128: "flux_1024"}[D]
    N = img[0] * img[1]
    inp = workloads.make_inputs(base, device="cuda", B=2, H=2, Nq=N, Nk=N)
    out, lse = fa.fwd_window(inp["q"], inp["k"], inp["v"], img[0], img[1], win[0], win[1],
                             shift[0], shift[1], scale=inp["scale"])
    torch.cuda.synchronize()
    assert fa.read_device_status() == 0
    q, k, v = (workloads.to_host_bits(inp[n]) for n in "qkv")
    o_ref, l_ref = oracle.window_attention(q, k, v, img[0], img[1], win[0], win[1], shift[0],
                                           shift[1], scale=inp["scale"])
    compare(out, lse, o_ref, l_ref, label=f"window D{D} {img} {win} {shift}")


def test_window_sd_latent_size():
    """SD1.5 512^2 latent grid (64x64 tokens, 8 heads of 64) with 8x8 shifted windows."""
    inp = workloads.make_inputs("sd_self", device="cuda")
    out, lse = fa.fwd_window(inp["q"], inp["k"], inp["v"], 64, 64, 8, 8, 4, 4, scale=inp["scale"])
    torch.cuda.synchronize()
    q, k, v = (workloads.to_host_bits(inp[n]) for n in "qkv")
    o_ref, l_ref = oracle.window_attention(q, k, v, 64, 64, 8, 8, 4, 4, scale=inp["scale"])
    compare(out, lse, o_ref, l_ref, label="window sd 64x64")


def test_window_validation():
    inp = workloads.make_inputs("sd_self", device="cuda", B=1, H=1, Nq=64, Nk=64)
    with pytest.raises(RuntimeError, match="INVALID_ARGUMENT"):
        fa.fwd_window(inp["q"], inp["k"], inp["v"], 8, 8, 3, 3)    # 3 does not divide 8



def test_window_is_one_launch_without_workspace(monkeypatch, capfd):
    """The windows are gathered and scattered by the attention kernel itself:
    one launch, no workspace (fa_window_workspace_bytes is 0)."""
    inp = workloads.make_inputs("sd_self", device="cuda", B=1, H=2)
    assert fa.window_workspace_bytes(1, 2, 64, 64, 64) == 0
    capfd.readouterr()
    monkeypatch.setenv("FA_LOG", "1")
    out, lse = fa.fwd_window(inp["q"], inp["k"], inp["v"], 64, 64, 8, 8, 4, 4, scale=inp["scale"])
    torch.cuda.synchronize()
    monkeypatch.delenv("FA_LOG")
    assert fa.read_device_status() == 0
    kernels = [ln for ln in capfd.readouterr().err.splitlines() if ln.startswith("[fa] fa_")]
    assert len(kernels) == 1 and "window rows" in kernels[0], kernels


def test_window_bitwise_deterministic():
    """Two runs of the same shifted-window launch give the same bits."""
    inp = workloads.make_inputs("sd_self", device="cuda", B=2, H=2)
    args = (inp["q"], inp["k"], inp["v"], 64, 64, 8, 8, 4, 4)
    o1, l1 = fa.fwd_window(*args, scale=inp["scale"])
    o2, l2 = fa.fwd_window(*args, scale=inp["scale"])
    torch.cuda.synchronize()
    assert fa.read_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
