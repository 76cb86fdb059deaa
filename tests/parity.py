"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on
the same seeded bf16 inputs and compare with the stated tolerances.

Tolerances (attention forward, bf16 in / bf16 out, fp32 softmax):
  O:   max |Δ| <= 2e-2 and mean |Δ| <= 2e-3 over every compared element;
  LSE: |Δ| <= 1e-3 · max(|LSE|, 1); rows with LSE = -inf must match exactly.
"""
import numpy as np
import torch

import oracle
import unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import workloads

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_REL = 1e-3


def run_gpu(inp, scale=None):
    scale = inp["scale"] if scale is None else scale
    out, lse = fa.fwd(inp["q"], inp["k"], inp["v"], mask=inp["mask"], scale=scale)
    torch.cuda.synchronize()
    assert fa.read_device_status() == 0, "kernel reported a wait timeout"
    return out, lse


def run_oracle(inp, scale=None, rows=None):
    scale = inp["scale"] if scale is None else scale
    mask = None if inp["mask"] is None else inp["mask"].cpu().numpy()
    q, k, v = (workloads.to_host_bits(inp[n]) for n in "qkv")
    return oracle.attention(q, k, v, mask=mask, scale=scale, rows=rows)


def compare(out, lse, o_ref, lse_ref, rows=None, label=""):
    """Compare GPU (out, lse) against the oracle; rows = [BH, nrows] sampled indices."""
    B, H, Nq, D = out.shape
    o = out.float().cpu().numpy()
    ls = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o = o.reshape(B * H, Nq, D)[np.arange(B * H)[:, None], rows].reshape(o_ref.shape)
        ls = ls.reshape(B * H, Nq)[np.arange(B * H)[:, None], rows].reshape(lse_ref.shape)
    assert np.all(np.isfinite(o)), f"{label}: non-finite O"
    err = np.abs(o - o_ref)
    ninf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(ls), ninf_ref), f"{label}: -inf LSE rows differ"
    fin = ~ninf_ref
    lerr = np.abs(ls[fin] - lse_ref[fin]) / np.maximum(np.abs(lse_ref[fin]), 1.0)
    stats = dict(o_max=float(err.max()), o_mean=float(err.mean()),
                 lse_rel=float(lerr.max()) if lerr.size else 0.0)
    assert stats["o_max"] <= O_MAX_ABS, f"{label}: O max-abs {stats}"
    assert stats["o_mean"] <= O_MEAN_ABS, f"{label}: O mean-abs {stats}"
    assert stats["lse_rel"] <= LSE_REL, f"{label}: LSE rel {stats}"
    return stats
