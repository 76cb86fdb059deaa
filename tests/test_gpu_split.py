"""GPU parity of the split-key forward (fa_fwd_split: per-range partial O/LSE,
then the LSE merge) against the fp64 oracle, through the C ABI."""
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


def run_split(inp, num_splits, scale=None):
    scale = inp["scale"] if scale is None else scale
    out, lse = fa.fwd_split(inp["q"], inp["k"], inp["v"], mask=inp["mask"], scale=scale,
                            num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa.read_device_status() == 0
    return out, lse


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("Nq,Nk,splits", [(1, 700, 3), (129, 1000, 2), (256, 1025, 8),
                                          (300, 257, 16), (77, 128, 4)])
def test_split_parity(D, Nq, Nk, splits):
    base = {32: "page_example", 64: "sd_self", 128: "flux_1024"}[D]
    inp = workloads.make_inputs(base, device="cuda", B=2, H=2, Nq=Nq, Nk=Nk)
    out, lse = run_split(inp, splits)
    o_ref, lse_ref = run_oracle(inp)
    compare(out, lse, o_ref, lse_ref, label=f"split{splits} D{D} Nq{Nq} Nk{Nk}")


def test_split_with_fully_masked_ranges():
    inp = workloads.make_inputs("sd_cross", device="cuda", B=3, H=2, Nq=200, Nk=1024)
    m = torch.zeros(3, 1024)
    m[0, 100:] = float("-inf")        # ranges past key 100 see only masked keys
    m[1, :] = float("-inf")           # every key masked
    m[2, 5] = -2.0
    inp["mask"] = m.cuda().contiguous()
    out, lse = run_split(inp, 8)
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    o_ref, lse_ref = run_oracle(inp)
    compare(out, lse, o_ref, lse_ref, label="split masked ranges")


def test_one_range_is_the_unsplit_forward():
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=3, Nq=500, Nk=900)
    o1, l1 = run_split(inp, 1)
    o0, l0 = run_gpu(inp)
    assert torch.equal(o1, o0) and torch.equal(l1, l0)


def test_more_splits_than_key_blocks():
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=2, Nq=256, Nk=300)
    out, lse = run_split(inp, 64)        # 3 key blocks -> 3 ranges
    o_ref, lse_ref = run_oracle(inp)
    compare(out, lse, o_ref, lse_ref, label="split clamp")


def test_long_keys_few_queries_full_size():
    """One head pair, 256 queries, HunyuanVideo-length keys: the low-occupancy
    shape split-key exists for; split count from the library's heuristic."""
    inp = workloads.make_inputs("hunyuan_720p", device="cuda", B=1, H=2, Nq=256, Nk=119056)
    splits = fa.split_count(1, 2, 256, 119056)
    assert splits > 1
    out, lse = run_split(inp, splits)
    o_ref, lse_ref = run_oracle(inp)
    compare(out, lse, o_ref, lse_ref, label=f"long keys split{splits}")


def test_flux_2048_split_sampled_rows():
    inp = workloads.make_inputs("flux_2048", device="cuda")
    B, H, Nq, Nk, D = inp["shape"]
    rows = workloads.sample_rows(Nq, B * H, 128, seed=5)
    out, lse = run_split(inp, 2)
    o_ref, lse_ref = run_oracle(inp, rows=rows)
    compare(out, lse, o_ref, lse_ref, rows=rows, label="flux_2048 split2")


def test_split_deterministic():
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=2, Nq=300, Nk=3000)
    o1, l1 = run_split(inp, 5)
    o2, l2 = run_split(inp, 5)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_workspace_validation():
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=1, Nq=128, Nk=1024)
    out = torch.empty_like(inp["q"])
    lse = torch.empty(1, 1, 128, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError, match="INVALID_ARGUMENT"):
        fa.fa_fwd_split(inp["q"], inp["k"], inp["v"], None, out, lse, 4, small)
    with pytest.raises(RuntimeError, match="INVALID_ARGUMENT"):
        fa.fa_fwd_split(inp["q"], inp["k"], inp["v"], None, out, lse, 4, None)
