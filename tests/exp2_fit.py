"""Remez (minimax relative error) fit of 2^f on [-1/2, 1/2] — the polynomial the
kernel uses for the share of its exponentials that run on the FMA pipe — and a
bit-exact float32 model of that FMA-pipe exp2 (range reduction by adding
1.5·2^23, polynomial, exponent-field add)."""
import numpy as np


def remez_exp2(deg=3, a=-0.5, b=0.5, iters=20):
    n = deg + 2
    x = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    grid = np.linspace(a, b, 40001)
    c = None
    for _ in range(iters):
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * 2 ** x[i]
        sol = np.linalg.solve(A, 2 ** x)
        c = sol[:deg + 1]
        err = (np.polyval(c[::-1], grid) - 2 ** grid) / 2 ** grid
        d = np.diff(err)
        cand = [0] + [i for i in range(1, len(grid) - 1) if (d[i - 1] > 0) != (d[i] > 0)] + [len(grid) - 1]
        pts = []
        for i in cand:
            if pts and np.sign(err[i]) == np.sign(err[pts[-1]]):
                if abs(err[i]) > abs(err[pts[-1]]):
                    pts[-1] = i
            else:
                pts.append(i)
        while len(pts) > n:
            pts.pop(0 if abs(err[pts[0]]) < abs(err[pts[-1]]) else -1)
        if len(pts) < n:
            break
        x = grid[pts]
    return c


def exp2_fma_model(x, coeffs):
    """float32 model of the kernel's FMA-pipe exp2 (round-to-nearest at each step)."""
    f32 = np.float32
    x = np.maximum(np.atleast_1d(np.asarray(x, dtype=f32)), f32(-126.0))
    rnd = f32(12582912.0)
    j = (x + rnd).astype(f32)
    n = (j - rnd).astype(f32)
    f = (x - n).astype(f32)          # fma(n, -1, x) is exact here
    c0, c1, c2, c3 = (f32(v) for v in coeffs)
    q = (f * c3 + c2).astype(f32)
    q = (q * f + c1).astype(f32)
    q = (q * f + c0).astype(f32)
    bits = q.view(np.uint32) + (j.view(np.uint32) << np.uint32(23))
    return bits.astype(np.uint32).view(f32)
