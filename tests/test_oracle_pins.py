"""Pins of the CPU oracle against facts the pages and the mathematics fix.

Each test names what pins it.  None of them re-derives the oracle's own
formula: they check printed agreement on the handbook's worked example, an
independent blocked online-softmax recurrence, closed forms, invariants and a
library special case.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from unet_fa_fwd_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split()
            out[key] = float(val)
    return out


def _rng(seed):
    return np.random.default_rng(seed)


def _randn(rng, *shape):
    return rng.standard_normal(shape).astype(np.float32)


def blocked_online_softmax(q, k, v, mask=None, scale=None, block_q=64, block_k=64):
    """fp64 blocked attention with the running (m, l, acc) recurrence.

    Follows the handbook's `blocked` example ("算子加速：注意力、编译与融合",
    section "注意力：从O(N²)显存到分块"): per query block, m starts at -inf and
    l, acc at 0; per key block m_new = max(m, rowmax s), p = exp(s - m_new),
    l = l·e^(m - m_new) + Σp, acc = acc·e^(m - m_new) + p·V_j; out = acc / l.
    Written independently of the oracle, with tails and an additive key mask.
    Returns (out, lse, peak score-tile bytes as fp32).
    """
    q = q.astype(np.float64)
    k = k.astype(np.float64)
    v = v.astype(np.float64)
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros_like(q)
    lse = np.zeros((B, H, Nq))
    peak = 0
    for i in range(0, Nq, block_q):
        qi = q[:, :, i:i + block_q]
        bq = qi.shape[2]
        m = np.full((B, H, bq, 1), -np.inf)
        l = np.zeros((B, H, bq, 1))
        acc = np.zeros((B, H, bq, D))
        for j in range(0, Nk, block_k):
            kj = k[:, :, j:j + block_k]
            s = (qi @ np.swapaxes(kj, -1, -2)) * scale
            if mask is not None:
                s = s + mask[:, None, None, j:j + block_k].astype(np.float64)
            m_new = np.maximum(m, s.max(-1, keepdims=True))
            # Rows with no finite score yet keep m = -inf; shift by 0 there.
            shift = np.where(np.isfinite(m_new), m_new, 0.0)
            p = np.exp(s - shift)
            corr = np.where(np.isfinite(m), np.exp(m - shift), 0.0)
            l = l * corr + p.sum(-1, keepdims=True)
            acc = acc * corr + p @ v[:, :, j:j + block_k]
            m = m_new
            peak = max(peak, s.size * 4)
        with np.errstate(invalid="ignore", divide="ignore"):
            out[:, :, i:i + block_q] = np.where(l > 0, acc / np.where(l > 0, l, 1.0), 0.0)
            lse[:, :, i:i + block_q] = np.where(l[..., 0] > 0, m[..., 0] + np.log(np.where(l[..., 0] > 0, l[..., 0], 1.0)), -np.inf)
    return out, lse, peak


# ---------------------------------------------------------------------------
# The handbook's worked example: naive, blocked and SDPA agree at atol 1e-5.
# ---------------------------------------------------------------------------

def test_worked_example_agreement():
    g = _read_kv("handbook_worked_example.txt")
    B, H, N, D = int(g["B"]), int(g["H"]), int(g["N"]), int(g["D"])
    inp = workloads.make_inputs("page_example", keep_fp32=True)
    q, k, v = inp["q32"], inp["k32"], inp["v32"]
    assert q.shape == (B, H, N, D)
    # Same draws as torch.manual_seed(0) followed by three randn calls.
    torch.manual_seed(int(g["seed"]))
    q_ref = torch.randn(B, H, N, D)
    assert torch.equal(q, q_ref)

    o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    # The page's naive form in fp32 (scores materialised, softmax, times v).
    s = (q @ k.transpose(-1, -2)) / D ** 0.5
    o_naive = s.softmax(-1) @ v
    o_sdpa = F.scaled_dot_product_attention(q, k, v)
    atol = g["atol"]
    assert np.allclose(o, o_naive.numpy(), atol=atol)
    assert np.allclose(o, o_sdpa.numpy(), atol=atol)
    o_blk, lse_blk, peak = blocked_online_softmax(q.numpy(), k.numpy(), v.numpy(),
                                                  block_q=int(g["block"]), block_k=int(g["block"]))
    assert np.max(np.abs(o - o_blk)) < 1e-12
    assert np.max(np.abs(lse - lse_blk)) < 1e-12
    # Printed memory figures: naive score buffer 1024 KB, blocked peak 64 KB (16x).
    assert s.numel() * 4 / 1024 == g["naive_scores_kb"]
    assert peak / 1024 == g["blocked_peak_kb"]
    assert (s.numel() * 4) / peak == g["ratio"]


# ---------------------------------------------------------------------------
# Blocked online softmax == plain definition, by brute force on tiny shapes.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("Nq,Nk,D,bq,bk", [
    (1, 1, 1, 1, 1), (2, 3, 4, 1, 2), (3, 17, 4, 2, 3), (17, 64, 32, 16, 16),
    (64, 65, 32, 64, 64), (130, 130, 4, 64, 16), (5, 130, 32, 3, 64),
])
@pytest.mark.parametrize("masked", [False, True])
def test_blocked_equals_definition(Nq, Nk, D, bq, bk, masked):
    rng = _rng(Nq * 1000 + Nk * 10 + D)
    B, H = 2, 3
    q, k, v = _randn(rng, B, H, Nq, D), _randn(rng, B, H, Nk, D), _randn(rng, B, H, Nk, D)
    mask = None
    if masked:
        valid = rng.integers(1, Nk + 1, size=B)
        mask = np.where(np.arange(Nk)[None, :] < valid[:, None], 0.0, -np.inf).astype(np.float32)
        mask[:, 0] = np.float32(rng.standard_normal())  # a finite nonzero additive entry
    scale = 0.37
    o, lse = oracle.attention(q, k, v, mask=mask, scale=scale)
    o_b, lse_b, _ = blocked_online_softmax(q, k, v, mask=mask, scale=scale, block_q=bq, block_k=bk)
    assert np.max(np.abs(o - o_b)) < 1e-12
    assert np.max(np.abs(lse - lse_b)) < 1e-12


# ---------------------------------------------------------------------------
# Closed forms and invariants.
# ---------------------------------------------------------------------------

def test_probability_rows_sum_to_one():
    """The p_j of the oracle's row function (the one every forward entry point
    runs) form a probability distribution, are 0 on masked keys, and weight the
    V rows into exactly the O row the forward returns."""
    rng = _rng(1)
    q, k, v = _randn(rng, 1, 2, 7, 16), _randn(rng, 1, 2, 33, 16), _randn(rng, 1, 2, 33, 16)
    mask = np.zeros((1, 33), np.float32)
    mask[0, 20:] = -np.inf
    o_all, lse_all = oracle.attention(q, k, v, mask=mask)
    for h in range(2):
        for i in range(7):
            p, o_row, lse = oracle.probs(q, k, v, 0, h, i, mask=mask)
            assert abs(p.sum() - 1.0) < 1e-12
            assert np.all(p >= 0)
            assert np.all(p[20:] == 0)
            assert np.array_equal(o_row, o_all[0, h, i]) and lse == lse_all[0, h, i]
            assert np.max(np.abs(p @ v[0, h].astype(np.float64) - o_row)) < 1e-12
    mask[0, :] = -np.inf
    p, o_row, lse = oracle.probs(q, k, v, 0, 1, 3, mask=mask)
    assert np.all(p == 0) and np.all(o_row == 0) and lse == -np.inf


@pytest.mark.parametrize("how", ["zero_q", "zero_scale"])
def test_uniform_scores_give_mean_of_valid_values(how):
    """q = 0 (or scale = 0): every score is equal, so O is the column mean of the
    unmasked V rows and LSE = ln(#unmasked keys)."""
    rng = _rng(2)
    B, H, Nq, Nk, D = 2, 2, 5, 40, 8
    q, k, v = _randn(rng, B, H, Nq, D), _randn(rng, B, H, Nk, D), _randn(rng, B, H, Nk, D)
    valid = [13, 40]
    mask = np.where(np.arange(Nk)[None, :] < np.array(valid)[:, None], 0.0, -np.inf).astype(np.float32)
    scale = 0.5
    if how == "zero_q":
        q[:] = 0
    else:
        scale = 0.0
    o, lse = oracle.attention(q, k, v, mask=mask, scale=scale)
    for b in range(B):
        mean = v[b, :, :valid[b]].astype(np.float64).mean(axis=1)  # [H, D]
        assert np.max(np.abs(o[b] - mean[:, None, :])) < 1e-12
        assert np.max(np.abs(lse[b] - math.log(valid[b]))) < 1e-12


def test_constant_value_rows():
    rng = _rng(3)
    q, k = _randn(rng, 1, 3, 9, 16), _randn(rng, 1, 3, 50, 16)
    c = _randn(rng, 16)
    v = np.broadcast_to(c, (1, 3, 50, 16)).copy()
    o, _ = oracle.attention(q, k, v)
    assert np.max(np.abs(o - c.astype(np.float64))) < 1e-12


def test_single_key():
    """Nk = 1: O = V_0 and LSE = scale·q·k_0 + mask (mask added after the scale)."""
    rng = _rng(4)
    q, k, v = _randn(rng, 1, 2, 6, 8), _randn(rng, 1, 2, 1, 8), _randn(rng, 1, 2, 1, 8)
    mask = np.array([[0.75]], np.float32)
    scale = 2.0
    o, lse = oracle.attention(q, k, v, mask=mask, scale=scale)
    assert np.array_equal(o, np.broadcast_to(v.astype(np.float64), o.shape))
    want = scale * np.einsum("bhid,bhjd->bhi", q.astype(np.float64), k.astype(np.float64)) + 0.75
    assert np.max(np.abs(lse - want)) < 1e-12


def test_two_keys_logistic():
    """Nk = 2: p_0 = 1 / (1 + e^(s_1 - s_0)), a logistic function of the score gap."""
    q = np.array([[[[1.0, 2.0]]]], np.float32)
    k = np.array([[[[0.5, -1.0], [2.0, 0.25]]]], np.float32)
    v = np.array([[[[3.0, -1.0], [-2.0, 4.0]]]], np.float32)
    scale = 0.5
    s0 = scale * (1.0 * 0.5 + 2.0 * -1.0)
    s1 = scale * (1.0 * 2.0 + 2.0 * 0.25)
    p0 = 1.0 / (1.0 + math.exp(s1 - s0))
    o, lse = oracle.attention(q, k, v, scale=scale)
    assert abs(o[0, 0, 0, 0] - (p0 * 3.0 + (1 - p0) * -2.0)) < 1e-14
    assert abs(o[0, 0, 0, 1] - (p0 * -1.0 + (1 - p0) * 4.0)) < 1e-14
    assert abs(lse[0, 0, 0] - (s1 + math.log1p(math.exp(s0 - s1)))) < 1e-14


def test_key_channel_offset_shift():
    """A constant per-channel offset δ on K shifts row i's scores by scale·q_i·δ:
    O is unchanged and LSE moves by exactly that amount (the K outlier
    channels of the FLUX 2048² workload)."""
    rng = _rng(5)
    B, H, Nq, Nk, D = 1, 2, 11, 37, 16
    q = np.round(_randn(rng, B, H, Nq, D) * 8) / 8
    k = np.round(_randn(rng, B, H, Nk, D) * 8) / 8
    v = _randn(rng, B, H, Nk, D)
    delta = np.zeros(D, np.float32)
    delta[[1, 7, 9, 12]] = [3.0, -2.5, 4.0, 1.5]
    scale = 0.25
    o0, l0 = oracle.attention(q, k, v, scale=scale)
    o1, l1 = oracle.attention(q, (k + delta).astype(np.float32), v, scale=scale)
    assert np.max(np.abs(o1 - o0)) < 1e-10
    shift = scale * (q.astype(np.float64) @ delta.astype(np.float64))
    assert np.max(np.abs(l1 - l0 - shift)) < 1e-10


def test_mask_constant_offset_moves_lse_only():
    """Adding c to every mask entry of a batch moves LSE by c (the mask is not
    scaled) and leaves O unchanged."""
    rng = _rng(6)
    q, k, v = _randn(rng, 2, 2, 4, 8), _randn(rng, 2, 2, 10, 8), _randn(rng, 2, 2, 10, 8)
    mask = (np.round(_randn(rng, 2, 10) * 8) / 8).astype(np.float32)  # mask + c stays exact
    c = np.array([[1.5], [-0.75]], np.float32)
    o0, l0 = oracle.attention(q, k, v, mask=mask, scale=3.0)
    o1, l1 = oracle.attention(q, k, v, mask=(mask + c).astype(np.float32), scale=3.0)
    assert np.max(np.abs(o1 - o0)) < 1e-12
    assert np.max(np.abs(l1 - l0 - c[:, :, None].astype(np.float64))) < 1e-12


def test_key_permutation_invariance():
    rng = _rng(7)
    q, k, v = _randn(rng, 2, 2, 6, 8), _randn(rng, 2, 2, 29, 8), _randn(rng, 2, 2, 29, 8)
    mask = np.where(rng.random((2, 29)) < 0.3, -np.inf, 0.0).astype(np.float32)
    perm = rng.permutation(29)
    o0, l0 = oracle.attention(q, k, v, mask=mask)
    o1, l1 = oracle.attention(q, k[:, :, perm].copy(), v[:, :, perm].copy(), mask=mask[:, perm].copy())
    assert np.max(np.abs(o1 - o0)) < 1e-12
    assert np.max(np.abs(l1 - l0)) < 1e-12


def test_large_logits_pick_argmax_value():
    """Scores 100x larger: no overflow, and when the top score leads the
    runner-up by more than 50 the output is that key's V row."""
    rng = _rng(8)
    q, k, v = _randn(rng, 1, 1, 8, 16) * 100, _randn(rng, 1, 1, 64, 16) * 100, _randn(rng, 1, 1, 64, 16)
    o, lse = oracle.attention(q, k, v, scale=1.0)
    s = q[0, 0].astype(np.float64) @ k[0, 0].astype(np.float64).T
    checked = 0
    for i in range(8):
        top2 = np.sort(s[i])[-2:]
        assert np.isfinite(lse[0, 0, i])
        assert abs(lse[0, 0, i] - top2[1]) < 1e-6 + abs(top2[1]) * 1e-12 or top2[1] - top2[0] < 50
        if top2[1] - top2[0] > 50:
            j = int(np.argmax(s[i]))
            assert np.max(np.abs(o[0, 0, i] - v[0, 0, j])) < 1e-12
            checked += 1
    assert checked > 0


def test_fully_masked_row():
    rng = _rng(9)
    q, k, v = _randn(rng, 2, 1, 3, 4), _randn(rng, 2, 1, 5, 4), _randn(rng, 2, 1, 5, 4)
    mask = np.zeros((2, 5), np.float32)
    mask[1, :] = -np.inf
    o, lse = oracle.attention(q, k, v, mask=mask)
    assert np.all(o[1] == 0) and np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(lse[0]))


def test_library_sdpa_special_case():
    """torch's fp64 scaled_dot_product_attention with an additive mask (a library routine)."""
    rng = _rng(10)
    B, H, Nq, Nk, D = 2, 3, 19, 45, 24
    q, k, v = _randn(rng, B, H, Nq, D), _randn(rng, B, H, Nk, D), _randn(rng, B, H, Nk, D)
    mask = np.where(np.arange(Nk)[None, :] < np.array([[30], [45]]), 0.0, -np.inf).astype(np.float32)
    mask[:, 3] = 0.5
    scale = 0.3
    o, lse = oracle.attention(q, k, v, mask=mask, scale=scale)
    tq, tk, tv = (torch.from_numpy(x).double() for x in (q, k, v))
    tm = torch.from_numpy(mask).double()[:, None, None, :]
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=tm, scale=scale)
    assert np.max(np.abs(o - ref.numpy())) < 1e-12
    ref_lse = torch.logsumexp(scale * tq @ tk.transpose(-1, -2) + tm, dim=-1)
    assert np.max(np.abs(lse - ref_lse.numpy())) < 1e-12


def test_bf16_bits_path_equals_fp32_path():
    inp = workloads.make_inputs("sd_cross", B=1, H=2, Nq=33, Nk=80)
    q, k, v = (workloads.to_host_bits(inp[n]) for n in "qkv")
    qf, kf, vf = (inp[n].float().numpy() for n in "qkv")
    mask = inp["mask"].numpy()
    o_bits, l_bits = oracle.attention(q, k, v, mask=mask, scale=inp["scale"])
    o_f, l_f = oracle.attention(qf, kf, vf, mask=mask, scale=inp["scale"])
    assert np.array_equal(o_bits, o_f) and np.array_equal(l_bits, l_f)


def test_rows_mode_matches_full():
    rng = _rng(11)
    q, k, v = _randn(rng, 1, 3, 50, 8), _randn(rng, 1, 3, 21, 8), _randn(rng, 1, 3, 21, 8)
    rows = workloads.sample_rows(50, 3, nrows=7, seed=3)
    o, l = oracle.attention(q, k, v)
    o_r, l_r = oracle.attention(q, k, v, rows=rows)
    for bh in range(3):
        assert np.array_equal(o_r[0, bh], o[0, bh, rows[bh]])
        assert np.array_equal(l_r[0, bh], l[0, bh, rows[bh]])


def test_thread_count_does_not_change_result():
    rng = _rng(12)
    q, k, v = _randn(rng, 1, 2, 31, 8), _randn(rng, 1, 2, 17, 8), _randn(rng, 1, 2, 17, 8)
    o1, l1 = oracle.attention(q, k, v, nthreads=1)
    o4, l4 = oracle.attention(q, k, v, nthreads=4)
    assert np.array_equal(o1, o4) and np.array_equal(l1, l4)


# ---------------------------------------------------------------------------
# Split-key merge: attention over disjoint key ranges, merged by the LSE rule,
# equals attention over all keys (the exchange step of ring attention,
# "FlashAttention原理与工业实战" §6.2) — exact up to rounding.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cuts", [[0, 40, 97], [0, 1, 2, 97], [0, 64, 65, 97], [0, 20, 50, 80, 97]])
def test_split_key_merge_is_exact(cuts):
    rng = _rng(13)
    B, H, Nq, Nk, D = 2, 2, 9, 97, 16
    q, k, v = _randn(rng, B, H, Nq, D), _randn(rng, B, H, Nk, D), _randn(rng, B, H, Nk, D)
    mask = np.zeros((B, Nk), np.float32)
    mask[1, 30:] = -np.inf          # batch 1: the later ranges are fully masked
    mask[0, 5] = 1.25
    o_full, l_full = oracle.attention(q, k, v, mask=mask, scale=0.3)
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        parts.append(oracle.attention(q, k[:, :, a:b].copy(), v[:, :, a:b].copy(),
                                      mask=mask[:, a:b].copy(), scale=0.3))
    lses = np.stack([l for _, l in parts])                 # [S, B, H, Nq]
    m = lses.max(axis=0)
    w = np.exp(lses - m)                                   # -inf ranges weigh 0
    lse = m + np.log(w.sum(axis=0))
    o = sum(wi[..., None] * oi for wi, (oi, _) in zip(w, parts)) / w.sum(axis=0)[..., None]
    assert np.max(np.abs(o - o_full)) < 1e-12
    assert np.max(np.abs(lse - l_full)) < 1e-12


# ---------------------------------------------------------------------------
# General masks and causal (the oracle's fa_oracle_fwd_ex).
# ---------------------------------------------------------------------------

def test_full_mask_broadcast_of_key_padding_is_the_same_function():
    rng = _rng(20)
    B, H, Nq, Nk, D = 2, 3, 7, 19, 8
    q, k, v = _randn(rng, B, H, Nq, D), _randn(rng, B, H, Nk, D), _randn(rng, B, H, Nk, D)
    kp = np.where(rng.random((B, Nk)) < 0.3, -np.inf, 0.0).astype(np.float32)
    kp[:, 0] = 0.5
    full = np.broadcast_to(kp[:, None, None, :], (B, 1, Nq, Nk)).copy()
    o1, l1 = oracle.attention(q, k, v, mask=kp)
    o2, l2 = oracle.attention_ex(q, k, v, full_mask=full)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_causal_closed_forms():
    """Causal (key j <= query i): row 0 sees only key 0, so O_0 = V_0 and
    LSE_0 = s_00; with q = 0 row i is the mean of V_0..V_i, LSE = ln(i+1)."""
    rng = _rng(21)
    B, H, N, D = 1, 2, 12, 8
    q, k, v = _randn(rng, B, H, N, D), _randn(rng, B, H, N, D), _randn(rng, B, H, N, D)
    o, l = oracle.attention_ex(q, k, v, causal=True, scale=0.5)
    assert np.array_equal(o[:, :, 0], v[:, :, 0].astype(np.float64))
    s00 = 0.5 * np.einsum("bhd,bhd->bh", q[:, :, 0].astype(np.float64), k[:, :, 0].astype(np.float64))
    assert np.max(np.abs(l[:, :, 0] - s00)) < 1e-12
    q0 = np.zeros_like(q)
    o, l = oracle.attention_ex(q0, k, v, causal=True)
    for i in range(N):
        assert np.max(np.abs(o[:, :, i] - v[:, :, :i + 1].astype(np.float64).mean(axis=2))) < 1e-12
        assert np.max(np.abs(l[:, :, i] - np.log(i + 1))) < 1e-12


@pytest.mark.parametrize("heads", [1, 3])
def test_general_masks_against_library_sdpa(heads):
    """torch fp64 SDPA (a library routine) with an additive [B,heads,Nq,Nk]
    mask, a boolean mask (keep = True) and is_causal."""
    rng = _rng(22 + heads)
    B, H, Nq, Nk, D = 2, 3, 11, 11, 16
    q, k, v = _randn(rng, B, H, Nq, D), _randn(rng, B, H, Nk, D), _randn(rng, B, H, Nk, D)
    add = (rng.standard_normal((B, heads, Nq, Nk)) * 2).astype(np.float32)
    keep = rng.random((B, heads, Nq, Nk)) > 0.3
    keep[..., 0] = True
    tq, tk, tv = (torch.from_numpy(x).double() for x in (q, k, v))
    # additive
    o, l = oracle.attention_ex(q, k, v, full_mask=add, scale=0.4)
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(add).double(), scale=0.4)
    assert np.max(np.abs(o - ref.numpy())) < 1e-12
    # boolean: masked_fill(mask == 0, -inf) is the additive 0 / -inf mask
    as_add = np.where(keep, 0.0, -np.inf).astype(np.float32)
    o, l = oracle.attention_ex(q, k, v, full_mask=as_add)
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(keep))
    assert np.max(np.abs(o - ref.numpy())) < 1e-12
    # causal
    o, l = oracle.attention_ex(q, k, v, causal=True)
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    assert np.max(np.abs(o - ref.numpy())) < 1e-12
    s = (tq @ tk.transpose(-1, -2)) / np.sqrt(D)
    s = s.masked_fill(torch.ones(Nq, Nk, dtype=torch.bool).triu(1), float("-inf"))
    assert np.max(np.abs(l - torch.logsumexp(s, -1).numpy())) < 1e-12


def test_ex_rows_mode_matches_full():
    rng = _rng(24)
    q, k, v = _randn(rng, 1, 2, 40, 8), _randn(rng, 1, 2, 33, 8), _randn(rng, 1, 2, 33, 8)
    add = _randn(rng, 1, 2, 40, 33)
    rows = workloads.sample_rows(40, 2, nrows=6, seed=9)
    o, l = oracle.attention_ex(q, k, v, full_mask=add, causal=True)
    o_r, l_r = oracle.attention_ex(q, k, v, full_mask=add, causal=True, rows=rows)
    for bh in range(2):
        assert np.array_equal(o_r[0, bh], o[0, bh, rows[bh]])
        assert np.array_equal(l_r[0, bh], l[0, bh, rows[bh]])


# ---------------------------------------------------------------------------
# Window / shifted-window attention (the oracle's fa_oracle_window).
# ---------------------------------------------------------------------------

def _grid_inputs(seed, B=1, H=2, img=(8, 12), D=8):
    rng = _rng(seed)
    N = img[0] * img[1]
    return [_randn(rng, B, H, N, D) for _ in range(3)]


def test_window_equal_to_image_is_full_attention():
    q, k, v = _grid_inputs(30)
    o, l = oracle.window_attention(q, k, v, 8, 12, 8, 12, shift_h=3, shift_w=5)
    o_f, l_f = oracle.attention(q, k, v)
    assert np.max(np.abs(o - o_f)) < 1e-12 and np.max(np.abs(l - l_f)) < 1e-12


def test_one_by_one_windows_attend_to_self():
    q, k, v = _grid_inputs(31)
    o, l = oracle.window_attention(q, k, v, 8, 12, 1, 1, scale=0.5)
    assert np.array_equal(o, v.astype(np.float64))
    s_ii = 0.5 * np.einsum("bhnd,bhnd->bhn", q.astype(np.float64), k.astype(np.float64))
    assert np.max(np.abs(l - s_ii)) < 1e-12


def test_unshifted_windows_are_independent_attention_problems():
    """Each 4x6 window, gathered into its own tensor, is plain attention."""
    q, k, v = _grid_inputs(32)
    o, l = oracle.window_attention(q, k, v, 8, 12, 4, 6)
    grid = np.arange(96).reshape(8, 12)
    for wr in range(2):
        for wc in range(2):
            idx = grid[wr * 4:(wr + 1) * 4, wc * 6:(wc + 1) * 6].reshape(-1)
            o_w, l_w = oracle.attention(q[:, :, idx].copy(), k[:, :, idx].copy(), v[:, :, idx].copy())
            assert np.max(np.abs(o[:, :, idx] - o_w)) < 1e-12
            assert np.max(np.abs(l[:, :, idx] - l_w)) < 1e-12


def test_shift_is_a_cyclic_roll_of_the_grid():
    """Shifted windows = roll the grid by (-sh, -sw), unshifted windows, roll back."""
    q, k, v = _grid_inputs(33)
    sh, sw = 2, 3
    o, l = oracle.window_attention(q, k, v, 8, 12, 4, 6, shift_h=sh, shift_w=sw)

    def roll(x, a, b):
        B, H, N, D = x.shape
        return np.roll(x.reshape(B, H, 8, 12, D), (a, b), axis=(2, 3)).reshape(B, H, N, D)

    o_r, l_r = oracle.window_attention(roll(q, -sh, -sw), roll(k, -sh, -sw), roll(v, -sh, -sw),
                                       8, 12, 4, 6)
    assert np.max(np.abs(o - roll(o_r, sh, sw))) < 1e-12
    assert np.max(np.abs(l - roll(l_r[..., None], sh, sw)[..., 0])) < 1e-12
    # a shift by whole windows regroups the same windows: same result
    o2, _ = oracle.window_attention(q, k, v, 8, 12, 4, 6, shift_h=4, shift_w=6)
    o0, _ = oracle.window_attention(q, k, v, 8, 12, 4, 6)
    assert np.max(np.abs(o2 - o0)) < 1e-12
