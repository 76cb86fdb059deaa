"""The FLOP and byte formulas used for the roofline, against the figures the handbook prints."""
import os

from unet_fa_fwd_gb300 import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GB = 1024 ** 3


def _rows(name, header=True):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return (rows[0], rows[1:]) if header else (None, rows)


def test_attn_bytes_table():
    _, rows = _rows("handbook_attn_bytes.txt", header=False)
    assert len(rows) == 4
    for name, n, dh, h, scores_gb, naive_gb, flash_gb in rows:
        n, dh, h = int(n), int(dh), int(h)
        scores = accounting.naive_score_bytes(1, h, n, n)
        flash = accounting.qkvo_bytes(1, h, n, n, dh)
        naive = 2 * scores + flash
        assert f"{scores / GB:.1f}" == scores_gb, name
        assert f"{naive / GB:.1f}" == naive_gb, name
        assert f"{flash / GB:.2f}" == flash_gb, name


def test_block_profile_attention_row():
    _, rows = _rows("handbook_block_profile.txt")
    n, d, peak, bw, gflop, mb, intensity, t_us = rows[0]
    n, d, peak, bw = int(n), int(d), float(peak), float(bw)
    heads, dh = 24, 128
    assert heads * dh == d
    flops = accounting.attention_flops(1, heads, n, n, dh)
    byts = accounting.qkvo_bytes(1, heads, n, n, dh)
    assert f"{flops / 1e9:.1f}" == gflop
    assert f"{byts / 2 ** 20:.0f}" == mb
    assert f"{flops / byts:.0f}" == intensity
    assert f"{max(flops / peak, byts / bw) * 1e6:.0f}" == t_us


def test_algorithmic_bytes_adds_lse_and_mask():
    b = accounting.algorithmic_bytes(2, 8, 4096, 80, 64, masked=True)
    assert b == 2 * 2 * 8 * 64 * (2 * 4096 + 2 * 80) + 4 * 2 * 8 * 4096 + 4 * 2 * 80
