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
