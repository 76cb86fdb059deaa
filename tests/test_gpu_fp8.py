"""GPU parity of the FP8 (e4m3 Q K^T, SageAttention-style) forward against the
fp64 oracle — the exact attention — with the FP8 error budget.

Budget: the inputs of Q K^T are rounded to e4m3, whose unit roundoff (2^-4) is
16x bf16's (2^-8); the bf16 forward's bounds scale by 12.5 for O (max |dO|
<= 0.25, mean |dO| <= 2e-2).  LSE is held to an absolute bound: each score
carries an error of standard deviation ~ 2^-4 * sqrt(2/3) ~ 0.05 for unit-
variance inputs at scale 1/sqrt(D), and LSE (a smooth maximum of the scores)
moves by at most the largest score error, so |dLSE| <= 0.3 (6 sigma over the
~1e5 rows of a test).
"""
import numpy as np
import pytest
import torch

import unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import workloads

from .parity import run_oracle

pytestmark = pytest.mark.gpu

O_MAX_ABS = 0.25
O_MEAN_ABS = 2e-2
LSE_ABS = 0.3


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.load_library()
    torch.cuda.set_device(0)
    yield


def compare_fp8(out, lse, o_ref, l_ref, rows=None, label=""):
    B, H, Nq, D = out.shape
    o = out.float().cpu().numpy()
    ls = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o = o.reshape(B * H, Nq, D)[np.arange(B * H)[:, None], rows].reshape(o_ref.shape)
        ls = ls.reshape(B * H, Nq)[np.arange(B * H)[:, None], rows].reshape(l_ref.shape)
    assert np.all(np.isfinite(o)), label
    assert np.array_equal(np.isneginf(ls), np.isneginf(l_ref)), label
    err = np.abs(o - o_ref)
    fin = np.isfinite(l_ref)
    lerr = np.abs(ls[fin] - l_ref[fin])
    assert err.max() <= O_MAX_ABS, f"{label}: O max {err.max()}"
    assert err.mean() <= O_MEAN_ABS, f"{label}: O mean {err.mean()}"
    assert lerr.max() <= LSE_ABS, f"{label}: LSE {lerr.max()}"


def run_fp8(inp):
    out, lse = fa.fwd_fp8(inp["q"], inp["k"], inp["v"], mask=inp["mask"], scale=inp["scale"])
    torch.cuda.synchronize()
    assert fa.read_device_status() == 0
    return out, lse


@pytest.mark.parametrize("name", ["page_example", "sd_self", "sd_cross", "flux_1024"])
def test_fp8_configs_full(name):
    inp = workloads.make_inputs(name, device="cuda")
    out, lse = run_fp8(inp)
    o_ref, l_ref = run_oracle(inp)
    compare_fp8(out, lse, o_ref, l_ref, label=name)


@pytest.mark.parametrize("name", ["flux_2048", "hunyuan_720p"])
def test_fp8_configs_sampled(name):
    inp = workloads.make_inputs(name, device="cuda")
    B, H, Nq, Nk, D = inp["shape"]
    rows = workloads.sample_rows(Nq, B * H, 256, seed=inp["workload"].seed)
    out, lse = run_fp8(inp)
    o_ref, l_ref = run_oracle(inp, rows=rows)
    compare_fp8(out, lse, o_ref, l_ref, rows=rows, label=name)


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (127, 129), (300, 80), (513, 1000)])
def test_fp8_small_shapes(D, Nq, Nk):
    base = {32: "page_example", 64: "sd_self", 128: "flux_1024"}[D]
    inp = workloads.make_inputs(base, device="cuda", B=2, H=3, Nq=Nq, Nk=Nk)
    out, lse = run_fp8(inp)
    o_ref, l_ref = run_oracle(inp)
    compare_fp8(out, lse, o_ref, l_ref, label=f"fp8 D{D} {Nq}x{Nk}")


def test_fp8_smoothing_removes_key_outliers():
    """Constant offsets of 30 on a few K channels: without the mean smoothing
    the e4m3 block scale would be set by the offsets and swamp the rest."""
    inp = workloads.make_inputs("flux_1024", device="cuda", H=2, Nq=512, Nk=2048)
    k = inp["k"].float()
    k[:, :, :, [3, 50, 77]] += 30.0
    inp["k"] = k.to(torch.bfloat16).contiguous()
    out, lse = run_fp8(inp)
    o_ref, l_ref = run_oracle(inp)
    compare_fp8(out, lse, o_ref, l_ref, label="outliers")


def test_fp8_close_to_bf16_path():
    inp = workloads.make_inputs("flux_1024", device="cuda", H=4)
    o8, l8 = run_fp8(inp)
    ob, lb = fa.fwd(inp["q"], inp["k"], inp["v"], scale=inp["scale"])
    torch.cuda.synchronize()
    assert (o8.float() - ob.float()).abs().max().item() <= O_MAX_ABS
    assert (l8 - lb).abs().max().item() <= LSE_ABS


def test_fp8_workspace_validation():
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=1, Nq=128, Nk=256)
    out = torch.empty_like(inp["q"])
    lse = torch.empty(1, 1, 128, device="cuda")
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError, match="INVALID_ARGUMENT"):
        fa.fa_fwd_fp8(inp["q"], inp["k"], inp["v"], None, out, lse, small)


def _host_fp32(t):
    bits = workloads.to_host_bits(t).astype(np.uint32) << 16
    return bits.view(np.float32)


@pytest.mark.parametrize("name,kw", [
    ("page_example", {}),
    ("sd_cross", {}),
    ("flux_1024", dict(H=2)),
    ("sd_self", dict(B=1, H=2, Nq=333, Nk=517)),   # ragged query and key tails
])
def test_fp8_matches_its_emulation(name, kw):
    """Beyond the budget against the exact attention: the FP8 path agrees with a
    CPU emulation of the same quantisation (mean smoothing, 128-row block scales,
    e4m3 round-to-nearest-even) to the bf16 forward's tolerances — the rounding of
    P to bf16 for P·V is the remaining difference."""
    from oracle import fp8 as fp8_oracle
    from .parity import compare
    inp = workloads.make_inputs(name, device="cuda", **kw)
    out, lse = run_fp8(inp)
    q, k, v = (_host_fp32(inp[n]) for n in "qkv")
    mask = None if inp["mask"] is None else inp["mask"].cpu().numpy()
    o_e, l_e = fp8_oracle.attention_fp8_emulated(q, k, v, mask=mask, scale=inp["scale"])
    compare(out, lse, o_e, l_e, label=f"fp8 vs emulation {name}")
