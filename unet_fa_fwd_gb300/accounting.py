"""Algorithmic FLOP and byte counts of one attention forward.

FLOP: 4·B·H·Nq·Nk·D — two contractions (Q·Kᵀ and P·V) of 2·Nq·Nk·D each.
This is the attention row of the handbook's ``block_profile`` DiT roofline
("算子加速：注意力、编译与融合", section "访存受限的小算子": 4·n·n·d).

Bytes: the flash form of the handbook's ``attn_bytes`` memory model (section
"注意力：从O(N²)显存到分块"): read Q, K, V once, write O once; the scores stay
on chip.  The fp32 LSE write and the fp32 key mask read are added here.
"""
from __future__ import annotations


def attention_flops(B: int, H: int, Nq: int, Nk: int, D: int) -> int:
    return 4 * B * H * Nq * Nk * D


def qkvo_bytes(B: int, H: int, Nq: int, Nk: int, D: int, elem: int = 2) -> int:
    """Q + K + V read and O written, as in the handbook's flash memory model."""
    return elem * B * H * D * (2 * Nq + 2 * Nk)


def algorithmic_bytes(B: int, H: int, Nq: int, Nk: int, D: int, masked: bool = False) -> int:
    """Q, K, V (bf16) read + O (bf16) and LSE (fp32) written + mask (fp32 [B,Nk]) read."""
    b = qkvo_bytes(B, H, Nq, Nk, D) + 4 * B * H * Nq
    if masked:
        b += 4 * B * Nk
    return b


def naive_score_bytes(B: int, H: int, Nq: int, Nk: int, elem: int = 2) -> int:
    """Size of one materialised N×N score tensor (the handbook's ``scores`` term)."""
    return elem * B * H * Nq * Nk
