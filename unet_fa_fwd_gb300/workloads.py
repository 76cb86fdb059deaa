"""Seeded synthetic inputs shaped like the attention layers the pages discuss.

This module holds input generation only — no attention arithmetic — so that
both the CUDA path and the CPU oracle can be fed the same bf16 bytes.

Shapes, by page:
  * ``page_example``  — "算子加速：注意力、编译与融合", worked example in section
    "注意力：从O(N²)显存到分块": torch seed 0, q, k, v = randn(1, 4, 256, 32)
    drawn in that order.
  * ``sd_self`` / ``sd_cross`` — SD1.5 UNet attention at 512² (64×64 = 4096
    latent tokens; "Step 3.7 Flash" §4 table), 8 heads of 64.  The
    cross-attention reads the 77 text tokens padded to 80, with an additive
    key-padding mask from per-batch valid lengths ("Step 3.7 Flash" §2.2:
    dynamic batching pads and masks).
  * ``flux_1024`` / ``flux_2048`` / ``hunyuan_720p`` — token counts and head
    shapes of the handbook's ``attn_bytes`` table (4608 / 16896 / 119056
    tokens, 24 heads of 128).  FLUX 2048² puts per-channel offsets on 4
    channels of K per head (the outlier channels the SageAttention section
    smooths away); HunyuanVideo scales all three by 0.5.

Values are N(0,1) fp32, rounded to bf16 (round-to-nearest-even) by torch.
Datasets and trained weights are not used; these synthetic tensors stand in
for the activations of the named models.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    D: int
    seed: int
    masked: bool = False          # additive fp32 key-padding mask [B, Nk]
    k_outliers: int = 0           # channels of K per head given a constant offset
    outlier_std: float = 3.0      # std of those offsets
    value_scale: float = 1.0      # multiplies q, k, v
    full_oracle: bool = True      # False: the oracle checks sampled rows only
    description: str = ""

    @property
    def BH(self) -> int:
        return self.B * self.H

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(D), as the fp32 value passed to the kernel."""
        return float(np.float32(1.0 / math.sqrt(self.D)))


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("page_example", 1, 4, 256, 256, 32, seed=0,
                 description="handbook worked example B1 H4 N256 D32, torch seed 0"),
        Workload("sd_self", 2, 8, 4096, 4096, 64, seed=1001,
                 description="SD1.5 512^2 UNet self-attention B2 H8 N4096 D64"),
        Workload("sd_cross", 2, 8, 4096, 80, 64, seed=1101, masked=True,
                 description="SD1.5 512^2 cross-attention Nq4096 Nk80 (77 padded) D64, key mask"),
        Workload("flux_1024", 1, 24, 4608, 4608, 128, seed=1002,
                 description="FLUX 1024^2 joint attention B1 H24 N4608 D128"),
        Workload("flux_2048", 1, 24, 16896, 16896, 128, seed=1003, k_outliers=4,
                 full_oracle=False,
                 description="FLUX 2048^2 joint attention B1 H24 N16896 D128, K outlier channels"),
        Workload("hunyuan_720p", 1, 24, 119056, 119056, 128, seed=1004, value_scale=0.5,
                 full_oracle=False,
                 description="HunyuanVideo 720p attention B1 H24 N119056 D128, inputs x0.5"),
    ]
}

# Order of the five configurations of the workload list (SD self and cross
# count as one configuration).
CONFIG_ORDER = ["page_example", "sd_self", "sd_cross", "flux_1024", "flux_2048", "hunyuan_720p"]


def _small_generator(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(seed)


def make_inputs(w: Workload | str, device: str | torch.device = "cpu", *, B: int | None = None,
                H: int | None = None, Nq: int | None = None, Nk: int | None = None,
                keep_fp32: bool = False) -> dict:
    """Build q, k, v (bf16, [B,H,N,D], contiguous) and the optional fp32 mask [B,Nk].

    ``B/H/Nq/Nk`` override the workload's sizes (smaller cases with the same
    value distribution).  ``keep_fp32`` also returns the fp32 tensors before
    rounding (the handbook's worked example runs in fp32).
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    B = B or w.B
    H = H or w.H
    Nq = Nq or w.Nq
    Nk = Nk or w.Nk
    D = w.D
    device = torch.device(device)

    if w.name == "page_example":
        # Same stream as torch.manual_seed(0); randn(q), randn(k), randn(v) on the CPU.
        g = _small_generator(w.seed)
        q, k, v = (torch.randn(B, H, Nq if i == 0 else Nk, D, generator=g) for i in range(3))
        q, k, v = q.to(device), k.to(device), v.to(device)
    else:
        g = torch.Generator(device=device).manual_seed(w.seed)
        q = torch.randn(B, H, Nq, D, generator=g, device=device, dtype=torch.float32)
        k = torch.randn(B, H, Nk, D, generator=g, device=device, dtype=torch.float32)
        v = torch.randn(B, H, Nk, D, generator=g, device=device, dtype=torch.float32)

    if w.k_outliers:
        gs = _small_generator(w.seed + 1)
        chans = torch.stack([torch.randperm(D, generator=gs)[: w.k_outliers] for _ in range(H)])
        offs = torch.randn(H, w.k_outliers, generator=gs) * w.outlier_std
        for h in range(H):
            for c, o in zip(chans[h].tolist(), offs[h].tolist()):
                k[:, h, :, c] += o

    if w.value_scale != 1.0:
        q.mul_(w.value_scale)
        k.mul_(w.value_scale)
        v.mul_(w.value_scale)

    mask = None
    valid = None
    if w.masked:
        gs = _small_generator(w.seed + 2)
        hi = min(77, Nk)
        lo = min(8, hi)
        valid = torch.randint(lo, hi + 1, (B,), generator=gs)
        cols = torch.arange(Nk)
        mask = torch.where(cols[None, :] < valid[:, None], 0.0, float("-inf")).to(torch.float32)
        mask = mask.to(device).contiguous()

    out = {
        "q": q.to(torch.bfloat16).contiguous(),
        "k": k.to(torch.bfloat16).contiguous(),
        "v": v.to(torch.bfloat16).contiguous(),
        "mask": mask,
        "valid_lengths": valid,
        "scale": w.scale,
        "workload": w,
        "shape": (B, H, Nq, Nk, D),
    }
    if keep_fp32:
        out.update(q32=q, k32=k, v32=v)
    return out


def sample_rows(Nq: int, BH: int, nrows: int = 512, seed: int = 0) -> np.ndarray:
    """Seeded query rows per head, int64 [BH, nrows].

    Each head gets row 0, row Nq-1 (the last, possibly partial, tile) and
    nrows-2 distinct rows drawn uniformly from the rest.  When Nq <= nrows
    every row is taken.
    """
    if Nq <= nrows:
        return np.tile(np.arange(Nq, dtype=np.int64), (BH, 1))
    if nrows == 1:
        return np.zeros((BH, 1), dtype=np.int64)
    rows = np.empty((BH, nrows), dtype=np.int64)
    for bh in range(BH):
        rng = np.random.default_rng([seed, bh])
        mid = rng.choice(np.arange(1, Nq - 1, dtype=np.int64), size=nrows - 2, replace=False)
        rows[bh] = np.concatenate([[0, Nq - 1], np.sort(mid)])
    return rows


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a host uint16 array (same bytes the GPU reads)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
