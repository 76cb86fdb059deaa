"""Failure detection on the GPU without a fault: a wait that nothing will
complete must end in FA_ERR_TIMEOUT read from the device status word, and the
context must stay usable.  FA_FAULT_INJECT=stall makes CTA 0's producer
withhold one K/V tile (the host-side hook); FA_WAIT_TIMEOUT_MS shortens every
bounded wait so the test takes a fraction of a second."""
import pytest
import torch

import oracle
import unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import workloads

from .parity import compare, run_oracle

pytestmark = pytest.mark.gpu


def test_withheld_tile_times_out_and_context_survives(monkeypatch):
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    fa.load_library()
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=2, Nq=512, Nk=1024)
    assert fa.read_device_status() == 0

    monkeypatch.setenv("FA_FAULT_INJECT", "stall")
    monkeypatch.setenv("FA_WAIT_TIMEOUT_MS", "100")
    out, lse = fa.fwd(inp["q"], inp["k"], inp["v"], scale=inp["scale"])   # enqueued: FA_OK
    torch.cuda.synchronize()                                             # no fault, no hang
    assert fa.read_device_status() == fa.binding.FA_ERR_TIMEOUT
    assert fa.read_device_status() == 0                                  # read resets the word

    monkeypatch.delenv("FA_FAULT_INJECT")
    monkeypatch.delenv("FA_WAIT_TIMEOUT_MS")
    out, lse = fa.fwd(inp["q"], inp["k"], inp["v"], scale=inp["scale"])
    torch.cuda.synchronize()
    assert fa.read_device_status() == 0
    o_ref, l_ref = run_oracle(inp)
    compare(out, lse, o_ref, l_ref, label="after timeout")


def test_withheld_tile_times_out_with_staged_mask(monkeypatch):
    """The same with a staged additive mask: the mask copier stops at the abort
    and waits for its own copies before the CTA exits."""
    torch.cuda.set_device(0)
    fa.load_library()
    inp = workloads.make_inputs("flux_1024", device="cuda", B=1, H=2, Nq=512, Nk=1024)
    g = torch.Generator(device="cuda").manual_seed(2)
    m = torch.randn(1, 1, 512, 1024, generator=g, device="cuda")
    assert fa.read_device_status() == 0

    monkeypatch.setenv("FA_FAULT_INJECT", "stall")
    monkeypatch.setenv("FA_WAIT_TIMEOUT_MS", "100")
    fa.fwd_ex(inp["q"], inp["k"], inp["v"], full_mask=m, scale=inp["scale"])
    torch.cuda.synchronize()
    assert fa.read_device_status() == fa.binding.FA_ERR_TIMEOUT

    monkeypatch.delenv("FA_FAULT_INJECT")
    monkeypatch.delenv("FA_WAIT_TIMEOUT_MS")
    out, lse = fa.fwd_ex(inp["q"], inp["k"], inp["v"], full_mask=m, scale=inp["scale"])
    torch.cuda.synchronize()
    assert fa.read_device_status() == 0
    q, k, v = (workloads.to_host_bits(inp[n]) for n in "qkv")
    o_ref, l_ref = oracle.attention_ex(q, k, v, full_mask=m.cpu().numpy(), scale=inp["scale"])
    compare(out, lse, o_ref, l_ref, label="staged mask after timeout")
