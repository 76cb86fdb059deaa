"""Pins for the FP8 emulation oracle (``oracle/fp8.py``), on the CPU.

The e4m3 rounding is pinned to the format's definition (every finite code is a
fixed point, midpoints go to the even neighbour, saturation at 448); the whole
emulation is pinned to the exact oracle on inputs that e4m3 represents exactly
(block max 448, zero-mean K), where quantisation changes nothing.
"""
import numpy as np
import pytest

import oracle
from oracle import fp8


def _e4m3_values():
    """All positive finite e4m3 values, ascending, with their 3-bit mantissa."""
    vals = [(m * 2.0 ** -9, m) for m in range(1, 8)]                 # subnormals
    for e in range(-6, 9):
        for m in range(8):
            if e == 8 and m == 7:
                continue                                             # S.1111.111 is NaN
            vals.append(((1 + m / 8) * 2.0 ** e, m))
    return vals


def test_every_finite_code_is_a_fixed_point():
    v = np.array([x for x, _ in _e4m3_values()])
    assert v.max() == 448.0 and v.min() == 2.0 ** -9 and len(v) == 7 + 15 * 8 - 1
    np.testing.assert_array_equal(fp8.e4m3_round(v), v)
    np.testing.assert_array_equal(fp8.e4m3_round(-v), -v)


def test_midpoints_round_to_even_mantissa():
    vals = _e4m3_values()
    for (a, ma), (b, mb) in zip(vals, vals[1:]):
        mid = (a + b) / 2
        want = a if ma % 2 == 0 else b
        assert fp8.e4m3_round(np.array([mid]))[0] == want, (a, b)
        # just off the midpoint goes to the nearer value
        assert fp8.e4m3_round(np.array([np.nextafter(mid, 0)]))[0] == a
        assert fp8.e4m3_round(np.array([np.nextafter(mid, 1e9)]))[0] == b


def test_rounding_examples_and_saturation():
    r = fp8.e4m3_round(np.array([0.0, 1.0, 0.1, 449.0, 464.0, 1e6, -1e6, 2.0 ** -10,
                                 3 * 2.0 ** -10, 2.0 ** -12]))
    # 0.1 = 12.8 steps of 2^-7 -> 13 steps; 2^-10 is the midpoint of 0 and 2^-9 -> 0 (even);
    # 1.5 * 2^-9 -> the even neighbour 2^-8
    np.testing.assert_array_equal(r, [0.0, 1.0, 13 * 2.0 ** -7, 448.0, 448.0, 448.0, -448.0, 0.0,
                                      2.0 ** -8, 0.0])


def _grid_inputs(seed, B=1, H=2, Nq=200, Nk=160, D=32):
    """Q and K on the e4m3 grid, each 128-row block holding 448, K with zero channel means."""
    rng = np.random.default_rng(seed)
    vals = np.array([x for x, _ in _e4m3_values()])
    small = vals[vals <= 8.0]
    def grid(shape):
        x = rng.choice(small, size=shape) * rng.choice([-1.0, 1.0], size=shape)
        return x
    q = grid((B, H, Nq, D))
    q[:, :, ::128, 0] = 448.0                       # every 128-row block reaches 448
    half = grid((B, H, Nk // 2, D))
    half[:, :, ::64, 1] = 448.0
    k = np.concatenate([half, -half], axis=2)       # rows k and -k: channel means exactly 0
    v = rng.standard_normal((B, H, Nk, D)).astype(np.float32)
    return q.astype(np.float32), k.astype(np.float32), v


def test_emulation_equals_exact_attention_on_representable_inputs():
    q, k, v = _grid_inputs(1)
    scale = 2.0 ** -17                              # scores of order one despite |x| <= 448
    o8, l8 = fp8.attention_fp8_emulated(q, k, v, scale=scale)
    o, l = oracle.attention(q, k, v, scale=scale)
    np.testing.assert_allclose(o8, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l8, l, rtol=1e-12, atol=1e-12)


def test_emulation_stays_within_the_fp8_budget():
    rng = np.random.default_rng(2)
    B, H, N, D = 1, 2, 300, 64
    q, k, v = (rng.standard_normal((B, H, N, D)).astype(np.float32) for _ in range(3))
    k += rng.standard_normal((1, H, 1, D)).astype(np.float32) * 3   # channel offsets (smoothed away)
    o8, l8 = fp8.attention_fp8_emulated(q, k, v)
    o, l = oracle.attention(q, k, v)
    assert np.abs(o8 - o).max() <= 0.25 and np.abs(o8 - o).mean() <= 2e-2
    assert np.abs(l8 - l).max() <= 0.3
    # and it is not the exact attention (quantisation is really applied)
    assert np.abs(o8 - o).max() > 1e-4


def test_fully_masked_row_in_emulation():
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((2, 1, 64, 32)).astype(np.float32) for _ in range(3))
    mask = np.zeros((2, 64), np.float32)
    mask[1, :] = -np.inf
    o8, l8 = fp8.attention_fp8_emulated(q, k, v, mask=mask)
    assert np.all(o8[1] == 0) and np.all(np.isneginf(l8[1]))
    assert np.all(np.isfinite(l8[0]))
