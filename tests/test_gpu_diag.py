"""GPU: the exponential-unit probe behind the benchmark's secondary (exp2) bound."""
import pytest
import torch

import unet_fa_fwd_gb300 as fa

pytestmark = pytest.mark.gpu


def test_ex2_rate_is_plausible():
    """One SM retires a small power-of-two number of ex2 per clock (16 or 32 on
    recent parts); the probe must land near such a rate, never above 64."""
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    rate = fa.measure_ex2_rate()
    assert 8.0 <= rate <= 64.0, rate
    # repeatable to a few percent
    again = fa.measure_ex2_rate()
    assert abs(again - rate) <= 0.05 * rate, (rate, again)


def test_launch_log(monkeypatch, capfd):
    """FA_LOG=1 describes each launch on stderr: kernel, tile, grid, smem, stages, units."""
    import torch
    import unet_fa_fwd_gb300 as fa
    from unet_fa_fwd_gb300 import workloads
    torch.cuda.set_device(0)
    inp = workloads.make_inputs("page_example", device="cuda")
    monkeypatch.setenv("FA_LOG", "1")
    fa.fwd(inp["q"], inp["k"], inp["v"], scale=inp["scale"])
    fa.fwd_split(inp["q"], inp["k"], inp["v"], scale=inp["scale"], num_splits=2)
    monkeypatch.delenv("FA_LOG")
    fa.fwd(inp["q"], inp["k"], inp["v"], scale=inp["scale"])
    torch.cuda.synchronize()
    err = capfd.readouterr().err
    lines = [ln for ln in err.splitlines() if ln.startswith("[fa] ")]
    # B1 H4 N256: 4 units of two query tiles on 4 CTAs; split: 8 units, then the merge
    assert len(lines) == 3, err
    assert "fa_fwd_kernel<D=32,bf16,mask none> tile 128x128 grid 4 x 384 threads" in lines[0]
    assert "units 4" in lines[0] and "key ranges 1" in lines[0] and "mask none" in lines[0]
    assert "grid 8 x 384" in lines[1] and "key ranges 2" in lines[1]
    assert lines[2].startswith("[fa] fa_merge_kernel<D=32>") and "2 ranges, 1024 rows" in lines[2]
