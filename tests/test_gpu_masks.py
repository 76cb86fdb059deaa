"""GPU parity of fa_fwd_ex (general additive / boolean masks, causal) against
the fp64 oracle's fa_oracle_fwd_ex, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import workloads

from .parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.load_library()
    torch.cuda.set_device(0)
    yield


def _inputs(D, B, H, Nq, Nk, seed=0):
    base = {32: "page_example", 64: "sd_self", 128: "flux_1024"}[D]
    return workloads.make_inputs(base, device="cuda", B=B, H=H, Nq=Nq, Nk=Nk)


def _oracle(inp, full_mask=None, key_mask=None, causal=False, rows=None):
    q, k, v = (workloads.to_host_bits(inp[n]) for n in "qkv")
    fm = None if full_mask is None else full_mask.cpu().numpy()
    km = None if key_mask is None else key_mask.cpu().numpy()
    return oracle.attention_ex(q, k, v, mask=km, full_mask=fm, causal=causal, scale=inp["scale"],
                               rows=rows)


def _run(inp, **kw):
    out, lse = fa.fwd_ex(inp["q"], inp["k"], inp["v"], scale=inp["scale"], **kw)
    torch.cuda.synchronize()
    assert fa.read_device_status() == 0
    return out, lse


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (127, 129), (256, 256), (300, 513), (513, 300)])
def test_causal(D, Nq, Nk):
    inp = _inputs(D, 2, 2, Nq, Nk)
    out, lse = _run(inp, causal=True)
    o_ref, l_ref = _oracle(inp, causal=True)
    compare(out, lse, o_ref, l_ref, label=f"causal D{D} {Nq}x{Nk}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("heads", [1, 2])
@pytest.mark.parametrize("Nq,Nk", [(130, 200), (256, 384), (200, 301)])
def test_additive_full_mask(D, heads, Nq, Nk):
    """Nk 200 / 384: 16-byte mask loads (8 keys at a time) with a ragged last
    block; Nk 301: rows not 16-byte aligned, scalar loads."""
    inp = _inputs(D, 2, 2, Nq, Nk)
    g = torch.Generator(device="cuda").manual_seed(5)
    m = torch.randn(2, heads, Nq, Nk, generator=g, device="cuda") * 2
    m[0, :, 3, :] = float("-inf")              # a fully masked row
    m[1, :, :, 7:20] = float("-inf")
    out, lse = _run(inp, full_mask=m.contiguous())
    o_ref, l_ref = _oracle(inp, full_mask=m)
    compare(out, lse, o_ref, l_ref, label=f"additive D{D} h{heads}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nk", [333, 336, 332])
def test_bool_mask(D, causal, Nk):
    """Nk 336: 8-byte mask loads; 333 and 332: rows not 8-byte aligned, scalar loads."""
    inp = _inputs(D, 1, 3, 200, Nk)
    g = torch.Generator(device="cuda").manual_seed(6)
    keep = torch.rand(1, 3, 200, Nk, generator=g, device="cuda") > 0.4
    keep[..., 0] = True
    out, lse = _run(inp, full_mask=keep.contiguous(), causal=causal)
    add = torch.where(keep, 0.0, float("-inf")).float()
    o_ref, l_ref = _oracle(inp, full_mask=add, causal=causal)
    compare(out, lse, o_ref, l_ref, label=f"bool D{D} causal{causal} Nk{Nk}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(300, 512), (513, 260), (129, 1000)])
def test_key_padding_with_causal(D, Nq, Nk):
    """Key-padding mask and the causal triangle together: Nk a multiple of 4
    (the mask values come from the lanes' shuffled loads) with valid lengths
    that cut blocks, and one batch entry whose padding covers whole blocks."""
    inp = _inputs(D, 2, 2, Nq, Nk)
    g = torch.Generator(device="cuda").manual_seed(9)
    km = torch.randn(2, Nk, generator=g, device="cuda")
    km[0, Nk - Nk // 3:] = float("-inf")
    km[1, 130:300] = float("-inf")
    out, lse = _run(inp, key_mask=km, causal=True)
    o_ref, l_ref = _oracle(inp, key_mask=km, causal=True)
    compare(out, lse, o_ref, l_ref, label=f"key mask + causal D{D} {Nq}x{Nk}")


def test_key_padding_through_ex_matches_fa_fwd():
    inp = workloads.make_inputs("sd_cross", device="cuda")
    o1, l1 = _run(inp, key_mask=inp["mask"])
    o0, l0 = fa.fwd(inp["q"], inp["k"], inp["v"], mask=inp["mask"], scale=inp["scale"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o0) and torch.equal(l1, l0)


def test_no_mask_through_ex_matches_fa_fwd():
    inp = workloads.make_inputs("flux_1024", device="cuda", H=3)
    o1, l1 = _run(inp)
    o0, l0 = fa.fwd(inp["q"], inp["k"], inp["v"], scale=inp["scale"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o0) and torch.equal(l1, l0)


def test_causal_flux_1024_full_size():
    inp = workloads.make_inputs("flux_1024", device="cuda")
    B, H, Nq, Nk, D = inp["shape"]
    rows = workloads.sample_rows(Nq, B * H, 256, seed=3)
    out, lse = _run(inp, causal=True)
    o_ref, l_ref = _oracle(inp, causal=True, rows=rows)
    compare(out, lse, o_ref, l_ref, rows=rows, label="causal flux_1024")


@pytest.mark.parametrize("D", [64, 128])
def test_causal_long_heads_run_head_by_head(D):
    """Causal with more query pairs per head than the grid has CTAs: units run
    head by head, heaviest first within a head (rows sampled from every region
    of the triangle, the ragged last tile included)."""
    G = torch.cuda.get_device_properties(0).multi_processor_count
    Nq = 256 * (G + 5) - 100
    inp = _inputs(D, 1, 2, Nq, Nq)
    rows = workloads.sample_rows(Nq, 2, 96, seed=4)  # rows 0 and Nq - 1 included
    out, lse = _run(inp, causal=True)
    o_ref, l_ref = _oracle(inp, causal=True, rows=rows)
    compare(out, lse, o_ref, l_ref, rows=rows, label=f"causal long heads D{D}")


def test_mask_validation():
    inp = _inputs(64, 1, 2, 64, 64)
    out = torch.empty_like(inp["q"])
    lse = torch.empty(1, 2, 64, device="cuda")
    bad_heads = torch.zeros(1, 3, 64, 64, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_fwd_ex(inp["q"], inp["k"], inp["v"], out, lse, full_mask=bad_heads)
    m = fa.FaMask if hasattr(fa, "FaMask") else None
    from unet_fa_fwd_gb300.binding import FaMask, load_library
    import ctypes
    lib = load_library()
    for kind, data, heads in [(7, 0x1000, 1), (2, None, 1), (2, 0x1002, 1), (3, 0x1000, 5)]:
        mk = FaMask(kind, data, heads)
        rc = lib.fa_fwd_ex(inp["q"].data_ptr(), inp["k"].data_ptr(), inp["v"].data_ptr(),
                           ctypes.byref(mk), 0, out.data_ptr(), lse.data_ptr(), 1, 2, 64, 64, 64,
                           ctypes.c_float(0.125), None)
        assert rc == 1, (kind, data, heads)


def test_causal_last_wave_single_tile_units():
    """Causal with pair units = SMs + 10: the last wave runs single-tile units,
    whose causal key limit is their own last row."""
    G = torch.cuda.get_device_properties(0).multi_processor_count
    inp = _inputs(64, 1, G // 2 + 5, 512, 512)
    out, lse = _run(inp, causal=True)
    o_ref, l_ref = _oracle(inp, causal=True)
    compare(out, lse, o_ref, l_ref, label="causal last-wave singles")


@pytest.mark.parametrize("kind", ["additive", "bool"])
def test_mask_base_not_vector_aligned(kind):
    """The C ABI admits an fp32 mask aligned to 4 bytes and a uint8 mask at any
    address: such masks take the scalar load path (no misaligned vector loads)."""
    Nq, Nk = 150, 256
    inp = _inputs(64, 1, 2, Nq, Nk)
    g = torch.Generator(device="cuda").manual_seed(9)
    if kind == "additive":
        buf = torch.empty(1 * 2 * Nq * Nk + 1, device="cuda", dtype=torch.float32)
        m = buf[1:].view(1, 2, Nq, Nk)            # base 4 bytes past a 256-byte boundary
        m.copy_(torch.randn(1, 2, Nq, Nk, generator=g, device="cuda"))
        ref_mask = m.clone()
    else:
        buf = torch.empty(1 * 2 * Nq * Nk + 3, device="cuda", dtype=torch.bool)
        m = buf[3:].view(1, 2, Nq, Nk)            # base 3 bytes past a 256-byte boundary
        m.copy_(torch.rand(1, 2, Nq, Nk, generator=g, device="cuda") > 0.3)
        m[..., 0] = True
        ref_mask = torch.where(m, 0.0, float("-inf")).float()
    assert m.data_ptr() % 16 != 0
    out, lse = _run(inp, full_mask=m)
    o_ref, l_ref = _oracle(inp, full_mask=ref_mask)
    compare(out, lse, o_ref, l_ref, label=f"{kind} mask, unaligned base")


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("kind", ["additive", "bool"])
@pytest.mark.parametrize("per_head", [False, True])
def test_staged_mask_many_units(D, kind, per_head):
    """Mask rows 16-byte aligned (Nk 1040): an fp32 mask is copied tile by
    tile into shared memory (a byte mask takes 16-byte loads).  More units than
    SMs, so a CTA runs several units (the mask pieces are counted across them);
    Nq 600 ends on a partial tile."""
    G = torch.cuda.get_device_properties(0).multi_processor_count
    B, H, Nq, Nk = 1, G // 2 + 7, 600, 1040
    inp = _inputs(D, B, H, Nq, Nk)
    g = torch.Generator(device="cuda").manual_seed(11)
    mh = H if per_head else 1
    if kind == "additive":
        m = torch.randn(B, mh, Nq, Nk, generator=g, device="cuda") * 2
        m[0, :, 5, :] = float("-inf")                 # a fully masked row
        m[0, :, 300:420, 128:300] = float("-inf")     # whole and partial masked blocks
        ref = m
    else:
        m = torch.rand(B, mh, Nq, Nk, generator=g, device="cuda") > 0.4
        m[..., 0] = True
        m[0, :, 300:420, 128:300] = False
        ref = torch.where(m, 0.0, float("-inf")).float()
    rows = workloads.sample_rows(Nq, B * H, 96, seed=D)
    out, lse = _run(inp, full_mask=m.contiguous())
    o_ref, l_ref = _oracle(inp, full_mask=ref, rows=rows)
    compare(out, lse, o_ref, l_ref, rows=rows, label=f"staged {kind} D{D} heads {mh}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(600, 1040), (1000, 400), (300, 900)])
def test_staged_additive_mask_with_causal(D, Nq, Nk):
    """A staged fp32 mask with the causal triangle: causal units stop at their
    last query row's key block, and the mask copier must walk the same
    shortened key ranges (Nq > Nk and Nq < Nk both)."""
    B, H = 2, 3
    inp = _inputs(D, B, H, Nq, Nk)
    g = torch.Generator(device="cuda").manual_seed(31)
    m = torch.randn(B, H, Nq, Nk, generator=g, device="cuda") * 1.5
    m[1, :, :, ::7] = float("-inf")
    out, lse = _run(inp, full_mask=m.contiguous(), causal=True)
    o_ref, l_ref = _oracle(inp, full_mask=m, causal=True)
    compare(out, lse, o_ref, l_ref, label=f"staged causal D{D} {Nq}x{Nk}")
