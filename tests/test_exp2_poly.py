"""The kernel's FMA-pipe exp2: coefficients come from a minimax fit, and the
float32 algorithm stays within the fit's error bound (far below the bf16
rounding the result then takes)."""
import os
import re

import numpy as np

from .exp2_fit import exp2_fma_model, remez_exp2

KERNEL = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "unet_fa_fwd_gb300", "csrc", "fa_fwd_kernel.cuh")


def kernel_coeffs():
    text = open(KERNEL, encoding="utf-8").read()
    vals = dict(re.findall(r"\b(c[0-3]) = ([0-9.eE+-]+)f", text))
    return [float(vals[f"c{i}"]) for i in range(4)]


def test_coefficients_are_the_minimax_fit():
    fit = remez_exp2(3).astype(np.float32)
    assert np.allclose(np.array(kernel_coeffs(), np.float32), fit, rtol=0, atol=2e-7)


def test_relative_error_bound():
    c = kernel_coeffs()
    x = np.linspace(-120.0, 8.0, 2_000_001, dtype=np.float32)
    got = exp2_fma_model(x, c).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got - want) / want
    assert rel.max() < 7.6e-5           # Remez bound 7.48e-5 plus fp32 evaluation
    assert rel.max() < 2.0 ** -9 / 20   # well below bf16 rounding of P


def test_integer_points_and_clamp():
    c = kernel_coeffs()
    for k in range(-125, 9):
        v = float(exp2_fma_model(np.float32(k), c)[0])
        assert abs(v / 2.0 ** k - 1) < 7.6e-5
    tiny = exp2_fma_model(np.array([-126.0, -300.0, -1e30], np.float32), c)
    assert np.all(tiny >= 0) and np.all(tiny < 2.0 ** -124)
