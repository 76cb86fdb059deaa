"""Seeded input generators: shapes, determinism and the stated value recipes."""
import numpy as np
import torch

from unet_fa_fwd_gb300 import workloads


def test_page_example_matches_manual_seed_stream():
    inp = workloads.make_inputs("page_example", keep_fp32=True)
    torch.manual_seed(0)
    q, k, v = (torch.randn(1, 4, 256, 32) for _ in range(3))
    assert torch.equal(inp["q32"], q) and torch.equal(inp["k32"], k) and torch.equal(inp["v32"], v)
    assert inp["q"].dtype == torch.bfloat16 and torch.equal(inp["q"], q.to(torch.bfloat16))


def test_deterministic_and_shaped():
    a = workloads.make_inputs("flux_1024", H=2, Nq=300, Nk=200)
    b = workloads.make_inputs("flux_1024", H=2, Nq=300, Nk=200)
    for n in "qkv":
        assert torch.equal(a[n], b[n])
        assert a[n].is_contiguous()
    assert a["q"].shape == (1, 2, 300, 128) and a["k"].shape == (1, 2, 200, 128)
    assert a["mask"] is None


def test_cross_attention_mask_recipe():
    inp = workloads.make_inputs("sd_cross")
    m = inp["mask"]
    assert m.shape == (2, 80) and m.dtype == torch.float32
    for b, L in enumerate(inp["valid_lengths"].tolist()):
        assert 8 <= L <= 77
        assert torch.all(m[b, :L] == 0) and torch.all(torch.isneginf(m[b, L:]))


def test_flux_2048_key_outlier_channels():
    w = workloads.WORKLOADS["flux_2048"]
    inp = workloads.make_inputs(w, H=3, Nq=8, Nk=4096)
    k = inp["k"].float()[0]                    # [H, Nk, D]
    mean = k.mean(dim=1)                       # per-channel mean over tokens
    for h in range(3):
        big = (mean[h].abs() > 0.3).sum().item()   # offsets ~N(0,3); token noise mean ~1/64
        assert 1 <= big <= w.k_outliers


def test_hunyuan_values_scaled():
    inp = workloads.make_inputs("hunyuan_720p", H=1, Nq=4096, Nk=4096)
    std = inp["v"].float().std().item()
    assert 0.45 < std < 0.55


def test_sample_rows():
    r = workloads.sample_rows(119056, 24, 512, seed=7)
    assert r.shape == (24, 512)
    assert np.all(r[:, 0] == 0) and np.all(r[:, 1] == 119055)
    for row in r:
        assert len(set(row.tolist())) == 512
    assert np.array_equal(r, workloads.sample_rows(119056, 24, 512, seed=7))
    small = workloads.sample_rows(100, 3, 512)
    assert small.shape == (3, 100)
