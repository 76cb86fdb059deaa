"""The debug build (libfa_fwd_debug.so, FA_DEBUG=1): every kernel checks its
unit schedule and the index of each global access, records the first
violation and skips the access.  Run in a child process (the library is
chosen when it is first loaded):

* the parity cases of every entry point — head dims 32/64/128, ragged Nq and
  Nk, key-padding / additive / boolean masks, causal, split keys, FP8, windows
  — must report no violation and still match the oracle;
* with a planted check (the O-store bound lowered by one row; the store's
  address is valid, only the check is tightened) the violation must be
  reported as FA_ERR_DEBUG_CHECK with the store check's id.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD_PARITY = r'''
import sys, torch
sys.path.insert(0, ROOT)
import oracle, unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import workloads
from tests.parity import compare, run_oracle
assert fa.debug_build(), "the debug library was not loaded"
torch.cuda.set_device(0)

def check(label, out, lse, o_ref, lse_ref):
    torch.cuda.synchronize()
    st = fa.read_device_status()
    rec = fa.debug_report()
    assert st == 0 and rec == [0] * 8, (label, st, rec)
    if o_ref is not None:
        compare(out, lse, o_ref, lse_ref, label=label)

for base, sizes in [("page_example", {}),
                    ("sd_self", dict(B=1, H=2, Nq=300, Nk=513)),
                    ("flux_1024", dict(B=1, H=2, Nq=257, Nk=1000)),
                    ("sd_cross", dict(B=2, H=2, Nq=384, Nk=80))]:
    inp = workloads.make_inputs(base, device="cuda", **sizes)
    out, lse = fa.fwd(inp["q"], inp["k"], inp["v"], mask=inp["mask"], scale=inp["scale"])
    check(base, out, lse, *run_oracle(inp))

inp = workloads.make_inputs("flux_1024", device="cuda", B=2, H=2, Nq=200, Nk=301)
qh, kh, vh = (workloads.to_host_bits(inp[n]) for n in "qkv")
g = torch.Generator(device="cuda").manual_seed(3)
add = torch.randn(2, 1, 200, 301, generator=g, device="cuda")
keep = torch.rand(2, 2, 200, 301, generator=g, device="cuda") > 0.2
for label, kw, okw in [
        ("additive", dict(full_mask=add), dict(full_mask=add.cpu().numpy())),
        ("bool", dict(full_mask=keep), dict(full_mask=torch.where(keep, 0.0, float("-inf")).cpu().numpy())),
        ("causal", dict(causal=True), dict(causal=True))]:
    out, lse = fa.fwd_ex(inp["q"], inp["k"], inp["v"], scale=inp["scale"], **kw)
    o_ref, l_ref = oracle.attention_ex(qh, kh, vh, scale=inp["scale"], **okw)
    check(label, out, lse, o_ref, l_ref)

inp = workloads.make_inputs("hunyuan_720p", device="cuda", B=1, H=2, Nq=256, Nk=4000)
out, lse = fa.fwd_split(inp["q"], inp["k"], inp["v"], scale=inp["scale"], num_splits=6)
check("split", out, lse, *run_oracle(inp))
out, lse = fa.fwd_fp8(inp["q"], inp["k"], inp["v"], scale=inp["scale"])
check("fp8", out, lse, None, None)

w = workloads.make_inputs("sd_self", device="cuda", B=1, H=2)
out, lse = fa.fwd_window(w["q"], w["k"], w["v"], 64, 64, 8, 8, 4, 4, scale=w["scale"])
o_ref, l_ref = oracle.window_attention(*(workloads.to_host_bits(w[n]) for n in "qkv"), 64, 64, 8, 8,
                                       4, 4, scale=w["scale"])
check("window", out, lse, o_ref, l_ref)
print("debug build: no violation")
'''

CHILD_PLANT = r'''
import sys, torch
sys.path.insert(0, ROOT)
import unet_fa_fwd_gb300 as fa
from unet_fa_fwd_gb300 import workloads
assert fa.debug_build()
torch.cuda.set_device(0)
inp = workloads.make_inputs("page_example", device="cuda")
fa.fwd(inp["q"], inp["k"], inp["v"], scale=inp["scale"])
torch.cuda.synchronize()
st = fa.read_device_status()
rec = fa.debug_report()
print("status", st, "record", rec)
assert st == fa.binding.FA_ERR_DEBUG_CHECK, st
assert rec[0] == 5 and rec[7] >= 1, rec
# the next call, without the plant, is clean again
'''


def _run(code, extra_env):
    env = dict(os.environ, FA_DEBUG="1", **extra_env)
    r = subprocess.run([sys.executable, "-c", code.replace("ROOT", repr(ROOT))], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return r.stdout


def test_debug_build_parity_cases_report_no_violation():
    out = _run(CHILD_PARITY, {})
    assert "no violation" in out


def test_debug_build_reports_a_planted_store_violation():
    out = _run(CHILD_PLANT, {"FA_DEBUG_PLANT": "store"})
    assert "status 5" in out
