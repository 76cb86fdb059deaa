"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Full oracle for the page example, SD1.5 self/cross and FLUX 1024²; 512 seeded
query rows per head (row 0 and the last row included) for FLUX 2048² and
HunyuanVideo 720p, in the same launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import workloads

from .parity import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.load_library()
    torch.cuda.set_device(0)
    yield


@pytest.mark.parametrize("name", ["page_example", "sd_self", "sd_cross", "flux_1024"])
def test_config_full(name):
    inp = workloads.make_inputs(name, device="cuda")
    out, lse = run_gpu(inp)
    o_ref, lse_ref = run_oracle(inp)
    s = compare(out, lse, o_ref, lse_ref, label=name)
    print(name, s)


@pytest.mark.parametrize("name", ["flux_2048", "hunyuan_720p"])
def test_config_sampled_rows(name):
    inp = workloads.make_inputs(name, device="cuda")
    B, H, Nq, Nk, D = inp["shape"]
    rows = workloads.sample_rows(Nq, B * H, 512, seed=inp["workload"].seed)
    out, lse = run_gpu(inp)
    o_ref, lse_ref = run_oracle(inp, rows=rows)
    s = compare(out, lse, o_ref, lse_ref, rows=rows, label=name)
    print(name, s)


SMALL = [(1, 1), (15, 127), (127, 129), (129, 15), (256, 256), (300, 80), (513, 1000), (1, 700)]


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("Nq,Nk", SMALL)
def test_small_shapes_and_tails(D, Nq, Nk):
    base = {32: "page_example", 64: "sd_self", 128: "flux_1024"}[D]
    inp = workloads.make_inputs(base, device="cuda", B=2, H=3, Nq=Nq, Nk=Nk)
    out, lse = run_gpu(inp)
    o_ref, lse_ref = run_oracle(inp)
    compare(out, lse, o_ref, lse_ref, label=f"D{D} Nq{Nq} Nk{Nk}")


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("Nk", [80, 200, 640, 77])
def test_key_padding_mask(D, Nk):
    inp = workloads.make_inputs("sd_cross", device="cuda", B=3, H=2, Nq=333, Nk=Nk)
    # widen the head dim by rebuilding q/k/v with the requested D
    g = torch.Generator(device="cuda").manual_seed(77 + D)
    for n, N in (("q", 333), ("k", Nk), ("v", Nk)):
        inp[n] = torch.randn(3, 2, N, D, generator=g, device="cuda").to(torch.bfloat16)
    valid = torch.tensor([8, min(77, Nk), Nk - 1])
    cols = torch.arange(Nk)
    m = torch.where(cols[None] < valid[:, None], 0.0, float("-inf"))
    m[0, 3] = -1.25          # a finite additive entry
    m[1, 0] = 0.5
    # batch entry 2: a distinct finite value on every valid key (a key-to-lane
    # mix-up in the vector path changes the result)
    m[2, : Nk - 1] = torch.linspace(-2.0, 1.5, Nk - 1)
    inp["mask"] = m.to(torch.float32).cuda().contiguous()
    inp["scale"] = float(np.float32(D ** -0.5))
    out, lse = run_gpu(inp)
    o_ref, lse_ref = run_oracle(inp)
    compare(out, lse, o_ref, lse_ref, label=f"mask D{D} Nk{Nk}")


def test_fully_masked_batch_gives_zero_and_neg_inf():
    inp = workloads.make_inputs("sd_cross", device="cuda", B=2, H=2, Nq=200, Nk=80)
    m = inp["mask"].clone()
    m[1, :] = float("-inf")
    inp["mask"] = m
    out, lse = run_gpu(inp)
    assert torch.all(out[1] == 0)
    assert torch.all(torch.isneginf(lse[1]))
    o_ref, lse_ref = run_oracle(inp)
    compare(out, lse, o_ref, lse_ref, label="fully masked")


@pytest.mark.parametrize("scale", [0.0, -0.125, 0.5])
def test_scale_values(scale):
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=2, Nq=257, Nk=300)
    out, lse = run_gpu(inp, scale=scale)
    o_ref, lse_ref = run_oracle(inp, scale=scale)
    compare(out, lse, o_ref, lse_ref, label=f"scale {scale}")


def test_large_logits_rescale_path():
    """Scores that grow along the key axis force repeated O rescaling."""
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=2, Nq=256, Nk=1024)
    ramp = torch.linspace(0.0, 6.0, 1024, device="cuda")[None, None, :, None]
    inp["k"] = (inp["k"].float() * 0.2 + ramp * inp["q"].float().mean(dim=2, keepdim=True)).to(
        torch.bfloat16).contiguous()
    inp["q"] = (inp["q"].float() * 4).to(torch.bfloat16).contiguous()
    out, lse = run_gpu(inp)
    o_ref, lse_ref = run_oracle(inp)
    compare(out, lse, o_ref, lse_ref, label="large logits")


def test_bitwise_deterministic():
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=4, Nq=1000, Nk=1500)
    o1, l1 = run_gpu(inp)
    o2, l2 = run_gpu(inp)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_invalid_arguments_launch_nothing():
    inp = workloads.make_inputs("page_example", device="cuda")
    q, k, v = inp["q"], inp["k"], inp["v"]
    out = torch.full_like(q, 7.0)
    lse = torch.full((1, 4, 256), 7.0, device="cuda")
    st = lambda **kw: fa.fa_fwd_status(*(kw.get(n, d) for n, d in [
        ("q", q.data_ptr()), ("k", k.data_ptr()), ("v", v.data_ptr()), ("mask", None),
        ("out", out.data_ptr()), ("lse", lse.data_ptr()), ("B", 1), ("H", 4), ("Nq", 256),
        ("Nk", 256), ("D", 32), ("scale", 0.1), ("stream", None)]))
    assert st(D=48) == 2
    assert st(q=None) == 1
    assert st(Nk=0) == 1
    assert st(scale=float("nan")) == 1
    assert st(out=q.data_ptr()) == 1
    assert st(q=q.data_ptr() + 2) == 1
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)


def _sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("D,Nk", [(64, 300), (128, 129)])
def test_last_wave_single_tile_units(D, Nk):
    """Pair units = SMs + 8: the last wave's 8 pairs run as 16 single-tile units."""
    G = _sm_count()
    base = {64: "sd_self", 128: "flux_1024"}[D]
    inp = workloads.make_inputs(base, device="cuda", B=1, H=G + 8, Nq=256, Nk=Nk)
    out, lse = run_gpu(inp)
    o_ref, lse_ref = run_oracle(inp)
    compare(out, lse, o_ref, lse_ref, label=f"last-wave singles D{D} Nk{Nk}")


def test_last_wave_single_tile_units_two_pairs_per_head():
    """Two pair units per head (Nq 512): the split pairs span the last heads' halves."""
    G = _sm_count()
    H = G // 2 + 5                     # pairs = G + 10, R = 10
    inp = workloads.make_inputs("sd_self", device="cuda", B=1, H=H, Nq=512, Nk=200)
    out, lse = run_gpu(inp)
    o_ref, lse_ref = run_oracle(inp)
    compare(out, lse, o_ref, lse_ref, label="last-wave singles Nq512")
