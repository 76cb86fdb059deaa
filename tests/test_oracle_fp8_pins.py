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


def _scaled_grid_blocks(rng, BH, N, D, exps, max_rows, negate_pairs=False):
    """[BH, N, D] with every 128-row block b on the e4m3 grid times 2^-exps[b] and its
    largest magnitude exactly 448 * 2^-exps[b], placed at row max_rows[b] of the block.
    With negate_pairs, the second 64 rows of each full block are the negatives of the
    first 64, so every block (and the whole tensor) has channel sums exactly 0."""
    vals = np.array([x for x, _ in _e4m3_values()])
    small = vals[vals <= 8.0]
    x = np.empty((BH, N, D))
    for b, e in enumerate(exps):
        r0, r1 = 128 * b, min(128 * (b + 1), N)
        n = r1 - r0
        half = n // 2 if negate_pairs else n
        blk = rng.choice(small, size=(BH, half, D)) * rng.choice([-1.0, 1.0], size=(BH, half, D))
        blk[:, max_rows[b] % half, b % D] = 448.0
        if negate_pairs:
            assert n % 2 == 0
            blk = np.concatenate([blk, -blk], axis=1)
        x[:, r0:r1] = blk * 2.0 ** -e
    return x


def test_block_scales_are_per_block_and_per_operand():
    """Q blocks with maxima 448·2^0, 448·2^-2, 448·2^-5 (the last block ragged) and K
    blocks with 448·2^-1, 448·2^-3: every block scale is a distinct power of two, so
    each block's scaled values land back on the e4m3 grid and quantisation is exact —
    but only if each 128-row block gets its own scale.  A wrong block size (the maxima
    sit in different 64-row halves), a wrong block index, or the Q and K scales
    swapped would round values off the grid or mis-scale scores, and the emulation
    would no longer equal the exact attention."""
    rng = np.random.default_rng(11)
    B, H, Nq, Nk, D = 1, 2, 300, 256, 32
    q = _scaled_grid_blocks(rng, B * H, Nq, D, exps=[0, 2, 5], max_rows=[3, 100, 40])
    k = _scaled_grid_blocks(rng, B * H, Nk, D, exps=[1, 3], max_rows=[70, 5], negate_pairs=True)
    q = q.reshape(B, H, Nq, D).astype(np.float32)
    k = k.reshape(B, H, Nk, D).astype(np.float32)
    v = rng.standard_normal((B, H, Nk, D)).astype(np.float32)
    assert np.all(k.astype(np.float64).sum(axis=2) == 0)        # smoothing is a no-op
    # the per-block scales the emulation derives are the planted powers of two
    _, sq = fp8._quantise_blocks(q.reshape(B * H, Nq, D))
    _, sk = fp8._quantise_blocks(k.reshape(B * H, Nk, D))
    np.testing.assert_array_equal(sq, np.tile([1.0, 2.0 ** -2, 2.0 ** -5], (B * H, 1)))
    np.testing.assert_array_equal(sk, np.tile([2.0 ** -1, 2.0 ** -3], (B * H, 1)))
    scale = 2.0 ** -12
    o8, l8 = fp8.attention_fp8_emulated(q, k, v, scale=scale)
    o, l = oracle.attention(q, k, v, scale=scale)
    np.testing.assert_allclose(o8, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l8, l, rtol=1e-12, atol=1e-12)


def test_mean_smoothing_lse_correction_is_exact():
    """K = K0 + c with K0 on the e4m3 grid (zero channel sums) and c an exactly
    representable per-channel offset: the emulation recovers c exactly as the mean,
    quantises K0 without error, and must add scale · q_i · c back to LSE — giving the
    exact attention's O and LSE to rounding (the offset moves every score of row i
    by the same scale · q_i · c, which the softmax ignores and LSE carries)."""
    rng = np.random.default_rng(12)
    B, H, Nq, Nk, D = 1, 2, 200, 256, 32
    q = _scaled_grid_blocks(rng, B * H, Nq, D, exps=[0, 1], max_rows=[9, 60])
    k0 = _scaled_grid_blocks(rng, B * H, Nk, D, exps=[2, 0], max_rows=[1, 33], negate_pairs=True)
    c = rng.integers(-12, 13, size=(B * H, 1, D)) * 0.25          # multiples of 1/4 in [-3, 3]
    c[:, 0, 0] = 2.75                                             # never all zero
    q = q.reshape(B, H, Nq, D).astype(np.float32)
    k = (k0 + c).reshape(B, H, Nk, D).astype(np.float32)
    assert np.array_equal(k.astype(np.float64), (k0 + c).reshape(B, H, Nk, D))   # exact in fp32
    v = rng.standard_normal((B, H, Nk, D)).astype(np.float32)
    scale = 2.0 ** -11
    o8, l8 = fp8.attention_fp8_emulated(q, k, v, scale=scale)
    o, l = oracle.attention(q, k, v, scale=scale)
    np.testing.assert_allclose(o8, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l8, l, rtol=1e-12, atol=1e-11)
    # the correction is really exercised: it moves LSE by far more than the tolerance
    shift = scale * np.einsum("hnd,hd->hn", q.reshape(B * H, Nq, D).astype(np.float64), c[:, 0])
    assert np.abs(shift).max() > 1e-2
