"""CPU emulation of the FP8 (e4m3) Q·Kᵀ forward — TEST INFRASTRUCTURE.

Only ``tests/`` may import this module.  The exact oracle (``oracle.attention``)
gives the attention the FP8 path approximates; this module gives what the FP8
path computes, step by step, so the GPU's quantisation can be checked tightly
rather than only inside the FP8 error budget.

Steps, in the order of "算子加速：注意力、编译与融合", section "SageAttention"
(smooth K by subtracting its mean, quantise Q and K, low-precision QKᵀ; P and V
stay 16-bit), with this build's choices where the section leaves them open:

1. mean_k[c] = (1/Nk) Σ_j k[j][c] per (b, h) and channel c;
2. K~ = K − mean_k (fp32);
3. per 128-row block of Q and of K~: s = max|x| / 448 (448 = largest finite
   e4m3), x8 = e4m3(x · (1/s)) with round-to-nearest-even and saturation;
4. S_ij = scale · s_q · s_k · Σ_c q8[i][c] k8[j][c] (+ mask), softmax, O = P·V
   in fp64 with the bf16 V;
5. LSE_i = ln Σ_j exp(S_ij) + scale · (q_i · mean_k) — the smoothing shifts every
   score of row i by that constant, which the softmax ignores and LSE adds back.

Steps 2–3 use fp32 arithmetic, as the device does; the rest is fp64.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even), saturating at ±448.

    e4m3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; normal binades
    2^-6 .. 2^8 with 8 steps each, subnormals in steps of 2^-9; the all-ones
    encoding of the top binade's last step is NaN, so 448 is the largest
    finite value.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.zeros_like(a)
    nz = a > 0
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    e = np.maximum(e, -6.0)                  # below 2^-6: subnormal steps of 2^-9
    quantum = np.exp2(e - 3.0)
    r = np.rint(a / quantum) * quantum       # np.rint rounds half to even
    out = np.where(nz, np.minimum(r, E4M3_MAX), 0.0)
    return np.copysign(out, x)


def _quantise_blocks(x32: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """x32: fp32 [BH, N, D].  Returns (e4m3 values as fp64 [BH, N, D], scales fp32 [BH, nblk])."""
    BH, N, D = x32.shape
    nblk = (N + 127) // 128
    q = np.empty(x32.shape, dtype=np.float64)
    scales = np.empty((BH, nblk), dtype=np.float32)
    for b in range(nblk):
        blk = x32[:, 128 * b:128 * (b + 1), :]
        amax = np.abs(blk).reshape(BH, -1).max(axis=1).astype(np.float32)
        s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        inv = (np.float32(1.0) / s).astype(np.float32)
        scaled = (blk * inv[:, None, None]).astype(np.float32)
        q[:, 128 * b:128 * (b + 1), :] = e4m3_round(scaled)
        scales[:, b] = s
    return q, scales


def attention_fp8_emulated(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                           mask: np.ndarray | None = None, scale: float | None = None):
    """q: [B,H,Nq,D], k, v: [B,H,Nk,D] as fp32 arrays holding bf16 values; mask fp32 [B,Nk].

    Returns (O, LSE) in fp64, as the FP8 forward computes them (see the module
    docstring for the steps)."""
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    q32 = np.asarray(q, dtype=np.float32).reshape(B * H, Nq, D)
    k32 = np.asarray(k, dtype=np.float32).reshape(B * H, Nk, D)
    v64 = np.asarray(v, dtype=np.float64).reshape(B * H, Nk, D)
    mean = (k32.astype(np.float64).sum(axis=1) / Nk).astype(np.float32)      # step 1
    ks = (k32 - mean[:, None, :]).astype(np.float32)                         # step 2
    q8, sq = _quantise_blocks(q32)                                           # step 3
    k8, sk = _quantise_blocks(ks)
    out = np.empty((B * H, Nq, D), dtype=np.float64)
    lse = np.empty((B * H, Nq), dtype=np.float64)
    rq = np.arange(Nq) // 128
    rk = np.arange(Nk) // 128
    for bh in range(B * H):
        raw = q8[bh] @ k8[bh].T                                              # step 4
        s = scale * raw * sq[bh][rq][:, None].astype(np.float64) * sk[bh][rk][None, :]
        if mask is not None:
            s = s + np.asarray(mask, dtype=np.float64)[bh // H][None, :]
        m = s.max(axis=1, keepdims=True)
        fin = np.isfinite(m[:, 0])
        mm = np.where(np.isfinite(m), m, 0.0)
        p = np.exp(s - mm)
        l = p.sum(axis=1)
        with np.errstate(divide="ignore", invalid="ignore"):
            out[bh] = np.where(l[:, None] > 0, (p @ v64[bh]) / l[:, None], 0.0)
            corr = scale * (q32[bh].astype(np.float64) @ mean[bh].astype(np.float64))  # step 5
            lse[bh] = np.where(fin & (l > 0), mm[:, 0] + np.log(l) + corr, -np.inf)
    return out.reshape(B, H, Nq, D), lse.reshape(B, H, Nq)
