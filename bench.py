#!/usr/bin/env python3
"""Benchmark of the attention forward: attention TFLOP/s on one GB300, next to
the fp64 CPU oracle.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl native|reference]
                    [--variant fwd|fp8|causal|key_mask|additive_mask|bool_mask|window]

A step is one attention forward (one kernel launch) over the whole workload,
inputs resident in device memory.  Default workload: HunyuanVideo 720p
attention, B1 H24 N119056 D128 bf16 — the largest of the page configurations
that fits one GPU (Q/K/V 2.2 GB, far larger than the 129 MB L2, so no flush is
needed between steps).  FLUX 2048² (B1 H24 N16896 D128) and the smaller
configurations are reported under "also".  Prints one JSON line on rank 0.

N > 1 (under torchrun) runs one independent replica per GPU — the path has no
exchange step — and reports the whole-job throughput (weak scaling).
``--impl reference`` times the CPU oracle instead, on a bounded sample of the
same workload.  ``--variant`` times another entry point as the step (for
profiling one path alone; the end-to-end leg and the "also" blocks are then
skipped): the FP8 Q K^T forward, causal attention, a key-padding mask (last
quarter of the keys excluded), a per-(query, key) additive fp32 or boolean mask
(broadcast over heads), or 8x8 window attention on a 64x64 token grid (the
workload must have 4096 tokens).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s and % of GB300 dense-bf16 peak (1 GPU), vs CPU oracle"
FALLBACK_BF16_TFLOPS = 1900.0
KERNEL_NAME = "fa_fwd_kernel"


# --------------------------------------------------------------------- helpers

KERNEL_FILES = ("fa_fwd_kernel.cuh", "fa_attn_impl.cuh", "fa_fastdiv.h", "sm100_ptx.cuh",
                "tmem_ldst.inc", "mma_batch.inc")


def kernel_source_hash() -> str:
    """sha256 over the files that define the attention kernel and its launch plan
    (device code, tensor-memory / MMA wrappers, unit schedule)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "unet_fa_fwd_gb300", "csrc")
    for name in KERNEL_FILES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return peaks, "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


def read_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel."""
    path = os.path.join(ROOT, "profiles", f"{KERNEL_NAME}_{workload}_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256") != kernel_source_hash():
            return None
        return int(float(kv["dram_bytes_per_launch"]))
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not self.lines:
            return None
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = max(smax, float(parts[1]))
            except ValueError:
                continue
            for n, p in zip(names, parts[3:7]):
                if p.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        busy = [s for s in sm if s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- distributed

def launches_per_step(step, device) -> int:
    """Kernels of this library one call of `step` launches, counted from the
    library's own launch log (FA_LOG=1 describes every launch on stderr; the
    descriptor is redirected to a temporary file for the one call)."""
    import re
    import tempfile
    import torch
    torch.cuda.synchronize(device)
    sys.stderr.flush()
    saved = os.dup(2)
    with tempfile.TemporaryFile() as f:
        os.dup2(f.fileno(), 2)
        os.environ["FA_LOG"] = "1"
        try:
            step()
            torch.cuda.synchronize(device)
        finally:
            os.environ.pop("FA_LOG", None)
            os.dup2(saved, 2)
            os.close(saved)
        f.seek(0)
        text = f.read().decode(errors="replace")
    return sum(len(re.findall(r"\bfa_\w+_kernel\b", ln))
               for ln in text.splitlines() if ln.startswith("[fa] "))


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, group=None, device=None) -> float:
    """Max of a per-rank float over the process group (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def whole_job_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Units processed by all ranks divided by the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------- CPU oracle

class OracleSampler:
    """The fp64 CPU oracle on seeded query rows of a workload (all keys per row)."""

    def __init__(self, inp, seed: int = 12345):
        import oracle
        from unet_fa_fwd_gb300 import workloads

        self.oracle, self.workloads = oracle, workloads
        self.inp = inp
        self.seed = seed
        self.shape = inp["shape"]
        self.mask = None if inp["mask"] is None else inp["mask"].cpu().numpy()
        self.qkv = [workloads.to_host_bits(inp[n]) for n in "qkv"]
        self.threads = oracle.default_threads()

    def run(self, rows_per_head: int):
        """Returns (flops, seconds, rows_per_head actually used)."""
        B, H, Nq, Nk, D = self.shape
        rows = self.workloads.sample_rows(Nq, B * H, rows_per_head, seed=self.seed)
        t0 = time.perf_counter()
        self.oracle.attention(*self.qkv, mask=self.mask, scale=self.inp["scale"], rows=rows,
                              nthreads=self.threads)
        dt = time.perf_counter() - t0
        return 4.0 * B * H * rows.shape[1] * Nk * D, dt, rows.shape[1]

    def rows_for(self, budget_s: float) -> int:
        """Rows per head whose oracle time is about budget_s (calibrated on one row per head)."""
        B, H, Nq, Nk, D = self.shape
        _, dt, r = self.run(2)
        per_row = dt / (r * B * H)
        return int(max(1, min(Nq, budget_s / max(per_row, 1e-9) / (B * H))))


# ---------------------------------------------------------------------- main

def bench_native(args, world, rank, local):
    import torch
    import torch.distributed as dist

    import unet_fa_fwd_gb300 as fa
    from unet_fa_fwd_gb300 import accounting, workloads

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    fa.load_library()

    w = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(w, device=device, H=args.heads)
    B, H, Nq, Nk, D = inp["shape"]
    q, k, v, mask = inp["q"], inp["k"], inp["v"], inp["mask"]
    out = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=device)
    flops = accounting.attention_flops(B, H, Nq, Nk, D)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v)) + (
        0 if mask is None else mask.numel() * 4)
    stream = torch.cuda.current_stream(device)

    variant = args.variant
    if variant == "fwd":
        def step():
            fa.fa_fwd(q, k, v, mask, out, lse, scale=inp["scale"], stream=stream)
    elif variant == "fp8":
        ws8v = torch.empty(fa.fp8_workspace_bytes(B, H, Nq, Nk, D), dtype=torch.uint8, device=device)

        def step():
            fa.fa_fwd_fp8(q, k, v, mask, out, lse, ws8v, scale=inp["scale"], stream=stream)
    elif variant == "causal":
        kept = Nq * (Nq + 1) // 2 if Nq <= Nk else Nk * (Nk + 1) // 2 + (Nq - Nk) * Nk
        flops = 4.0 * B * H * D * kept

        def step():
            fa.fa_fwd_ex(q, k, v, out, lse, causal=True, scale=inp["scale"], stream=stream)
    elif variant == "key_mask":
        kmask = torch.zeros((B, Nk), dtype=torch.float32, device=device)
        kmask[:, Nk - Nk // 4:] = float("-inf")
        in_bytes += kmask.numel() * 4

        def step():
            fa.fa_fwd_ex(q, k, v, out, lse, key_mask=kmask, scale=inp["scale"], stream=stream)
    elif variant in ("additive_mask", "bool_mask"):
        g = torch.Generator(device=device).manual_seed(2024)
        if variant == "additive_mask":
            fmask = torch.randn((B, 1, Nq, Nk), generator=g, device=device, dtype=torch.float32)
        else:
            fmask = torch.rand((B, 1, Nq, Nk), generator=g, device=device) > 0.1
        in_bytes += fmask.numel() * fmask.element_size()

        def step():
            fa.fa_fwd_ex(q, k, v, out, lse, full_mask=fmask, scale=inp["scale"], stream=stream)
    elif variant == "window":
        if Nq != 4096 or Nk != 4096:
            raise SystemExit("--variant window needs a 4096-token workload (64x64 grid)")
        flops = 4.0 * B * H * Nq * 64 * D

        def step():
            fa.fwd_window(q, k, v, 64, 64, 8, 8, 0, 0, scale=inp["scale"], stream=stream)
    else:
        raise SystemExit(f"unknown variant {variant}")

    def time_steps(fn, n):
        """Mean device time (ms) of n back-to-back calls after 2 warm-up calls."""
        for _ in range(2):
            fn()
        torch.cuda.synchronize(device)
        t0_, t1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0_.record(stream)
        for _ in range(n):
            fn()
        t1_.record(stream)
        torch.cuda.synchronize(device)
        if fa.read_device_status(stream) != 0:
            raise RuntimeError("kernel wait timed out")
        return t0_.elapsed_time(t1_) / n

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    kernels_per_step = launches_per_step(step, device)
    if fa.read_device_status(stream) != 0:
        raise RuntimeError("kernel wait timed out during warm-up")

    # ---- device-resident timed region ----
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(device)
        e0.record(stream)
        for i in range(args.steps):
            step()
            step_ev[i].record(stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        if world > 1:
            dist.barrier()
    secs = e0.elapsed_time(e1) / 1e3
    # per-step device times (an event after every launch; the first pairs with e0)
    step_ms = [e0.elapsed_time(step_ev[0])] + [step_ev[i - 1].elapsed_time(step_ev[i])
                                               for i in range(1, args.steps)]
    max_secs = max_over_ranks(secs, device=device)
    if fa.read_device_status(stream) != 0:
        raise RuntimeError("kernel wait timed out in the timed region")
    value_tflops = whole_job_throughput(flops * args.steps, world, max_secs) / 1e12
    ms_per_step = max_secs * 1e3 / args.steps
    kernel_tflops = flops / (ms_per_step / 1e3) / 1e12

    # ---- end to end: pinned host inputs -> device -> fa_fwd -> host outputs ----
    # Every step uploads its Q/K/V (and mask) from pinned host memory, runs the
    # forward through the C ABI and downloads O and LSE.  Two buffer sets and
    # four streams (Q upload, K/V upload, compute, download) let step i+1's
    # uploads and step i-1's download overlap step i's kernel (events keep each
    # buffer's writes after its previous reads).
    if variant != "fwd":
        args.also = False
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hmask = None if mask is None else mask.cpu().pin_memory()
    nbuf = 2
    dins = [[torch.empty_like(t) for t in (q, k, v)] + [None if mask is None else torch.empty_like(mask)]
            for _ in range(nbuf)]
    douts = [(torch.empty_like(out), torch.empty_like(lse)) for _ in range(nbuf)]
    houts = [(torch.empty(out.shape, dtype=out.dtype, pin_memory=True),
              torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)) for _ in range(nbuf)]
    s_in, s_in2, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    tev = lambda: torch.cuda.Event(enable_timing=True)
    in_done = [ev() for _ in range(nbuf)]
    in_done2 = [ev() for _ in range(nbuf)]
    up_events = []   # (start, end of Q, end of K/V) per timed step
    used = [ev() for _ in range(nbuf)]
    out_done = [ev() for _ in range(nbuf)]
    for i in range(nbuf):   # every buffer starts free
        used[i].record(stream)
        out_done[i].record(stream)

    def e2e_step(i, timed=False):
        b = i % nbuf
        dq, dk, dv, dm = dins[b]
        do, dl = douts[b]
        ho, hl = houts[b]
        marks = (tev(), tev(), tev()) if timed else None
        with torch.cuda.stream(s_in):
            s_in.wait_event(used[b])
            s_in2.wait_event(used[b])
            if timed:
                marks[0].record(s_in)
                s_in2.wait_event(marks[0])
            dq.copy_(hq, non_blocking=True)
            if dm is not None:
                dm.copy_(hmask, non_blocking=True)
            in_done[b].record(s_in)
            if timed:
                marks[1].record(s_in)
        with torch.cuda.stream(s_in2):
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            in_done2[b].record(s_in2)
            if timed:
                marks[2].record(s_in2)
        if timed:
            up_events.append(marks)
        stream.wait_event(in_done[b])
        stream.wait_event(in_done2[b])
        stream.wait_event(out_done[b])
        fa.fa_fwd(dq, dk, dv, dm, do, dl, scale=inp["scale"], stream=stream)
        used[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(used[b])
            ho.copy_(do, non_blocking=True)
            hl.copy_(dl, non_blocking=True)
            out_done[b].record(s_out)

    e2e_steps = max(10, args.steps // 10) if variant == "fwd" else 0
    e2e_secs = 0.0
    if e2e_steps:
        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(device)
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(i, timed=True)
        torch.cuda.synchronize(device)
        e2e_secs = max_over_ranks(time.perf_counter() - t0, device=device)
    # achieved host-to-device rate: bytes of one step's uploads over the time
    # from their start to the later of the two streams' ends (median over steps)
    up_ms = [max(m0.elapsed_time(m1), m0.elapsed_time(m2)) for m0, m1, m2 in up_events]
    h2d_gbs = in_bytes / (statistics.median(up_ms) * 1e6) if up_ms else 0.0
    e2e_tflops = (whole_job_throughput(flops * e2e_steps, world, e2e_secs) / 1e12
                  if e2e_steps else 0.0)
    out_bytes = out.numel() * 2 + lse.numel() * 4
    del dins, douts

    # ---- the other large workload (few steps each), bf16 and FP8 Q K^T ----
    also = {}
    if args.also and rank == 0:
        del hq, hk, hv, houts
        other = "flux_2048" if args.workload != "flux_2048" else "hunyuan_720p"
        hw = workloads.make_inputs(other, device=device)
        hB, hH, hNq, hNk, hD = hw["shape"]
        hoAll = torch.empty_like(hw["q"])
        hl = torch.empty((hB, hH, hNq), dtype=torch.float32, device=device)
        hfl = accounting.attention_flops(hB, hH, hNq, hNk, hD)
        n_h = 20 if other == "flux_2048" else 5
        with ClockSampler(local) as hclocks:
            hms = time_steps(lambda: fa.fa_fwd(hw["q"], hw["k"], hw["v"], None, hoAll, hl,
                                               scale=hw["scale"], stream=stream), n_h)
        ws8o = torch.empty(fa.fp8_workspace_bytes(hB, hH, hNq, hNk, hD), dtype=torch.uint8,
                           device=device)
        hms8 = time_steps(lambda: fa.fa_fwd_fp8(hw["q"], hw["k"], hw["v"], None, hoAll, hl, ws8o,
                                                scale=hw["scale"], stream=stream), n_h)
        also[other] = {"ms_per_step": round(hms, 4), "tflops": round(hfl / hms / 1e9, 1),
                       "steps": n_h, "clocks": hclocks.summary(),
                       "fp8_qk": {"ms_per_step": round(hms8, 4),
                                  "tflops": round(hfl / hms8 / 1e9, 1),
                                  "speedup_vs_bf16": round(hms / hms8, 3),
                                  "note": "pre-pass included; bf16-equivalent FLOPs"}}
        del hw, hoAll, hl, ws8o

    # ---- the page's smaller configurations, each launch timed alone after an L2 flush ----
    if args.also and rank == 0:
        # the long loops above leave the GPU at its power cap; idle briefly so the
        # short launches below run at the clocks a cold start sees
        time.sleep(3.0)
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)  # > 129 MB L2
        hbm = float(read_peaks()[0].get("hbm_gbs", 6671.5))
        small = {}
        for name in ("page_example", "sd_self", "sd_cross", "flux_1024"):
            w_in = workloads.make_inputs(name, device=device)
            sB, sH, sNq, sNk, sD = w_in["shape"]
            so_ = torch.empty_like(w_in["q"])
            sl_ = torch.empty((sB, sH, sNq), dtype=torch.float32, device=device)
            call = lambda: fa.fa_fwd(w_in["q"], w_in["k"], w_in["v"], w_in["mask"], so_, sl_,
                                     scale=w_in["scale"], stream=stream)
            for _ in range(3):
                call()
            times = []
            for _ in range(30):
                flush.zero_()
                c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c0.record(stream)
                call()
                c1.record(stream)
                torch.cuda.synchronize(device)
                times.append(c0.elapsed_time(c1))
            med = statistics.median(times)
            sfl = accounting.attention_flops(sB, sH, sNq, sNk, sD)
            sby = accounting.algorithmic_bytes(sB, sH, sNq, sNk, sD, masked=w_in["mask"] is not None)
            small[name] = {"ms_median": round(med, 4), "ms_min": round(min(times), 4),
                           "ms_max": round(max(times), 4), "tflops": round(sfl / med / 1e9, 1),
                           "hbm_gbs": round(sby / med / 1e6, 1),
                           "hbm_frac": round(sby / med / 1e6 / hbm, 4)}
            if name in ("page_example", "sd_cross"):
                # launch-bound sizes: also 1000 launches back to back (inputs L2-resident)
                b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                b0.record(stream)
                for _ in range(1000):
                    call()
                b1.record(stream)
                torch.cuda.synchronize(device)
                small[name]["us_per_launch_back_to_back"] = round(b0.elapsed_time(b1), 3)
            del w_in, so_, sl_
        also["small_configs"] = {"l2": "flushed (256 MB write) before every timed launch; "
                                       "us_per_launch_back_to_back: 1000 launches, L2-resident",
                                 "launches": 30, "configs": small}
        del flush

    # ---- causal, a general additive mask and window attention (warm, back to back) ----
    def time_call(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        t0_, t1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0_.record(stream)
        for _ in range(n):
            fn()
        t1_.record(stream)
        torch.cuda.synchronize(device)
        if fa.read_device_status(stream) != 0:
            raise RuntimeError("kernel wait timed out")
        return t0_.elapsed_time(t1_) / n

    if args.also and rank == 0:
        ext = {}
        # The short masked and window timings first, after a pause that lets the
        # clocks recover from the legs before (the long causal run heats the GPU).
        time.sleep(2.0)
        # additive fp32 mask [B, 1, Nq, Nk] (broadcast over heads) at FLUX 1024^2
        wm = workloads.make_inputs("flux_1024", device=device)
        mB, mH, mNq, mNk, mD = wm["shape"]
        g = torch.Generator(device=device).manual_seed(2024)
        fmask = torch.randn((mB, 1, mNq, mNk), generator=g, device=device, dtype=torch.float32)
        om_ = torch.empty_like(wm["q"])
        lm_ = torch.empty((mB, mH, mNq), dtype=torch.float32, device=device)
        with ClockSampler(local) as mclocks:
            msm = time_call(lambda: fa.fa_fwd_ex(wm["q"], wm["k"], wm["v"], om_, lm_, full_mask=fmask,
                                                 scale=wm["scale"], stream=stream), 20)
        ext["additive_mask"] = {"workload": "flux_1024", "mask": "fp32 [B,1,Nq,Nk] N(0,1)",
                                "ms_per_step": round(msm, 4),
                                "tflops": round(accounting.attention_flops(mB, mH, mNq, mNk, mD)
                                                / msm / 1e9, 1),
                                "mask_mb": round(fmask.numel() * 4 / 1e6, 1),
                                "clocks": mclocks.summary()}
        del wm, fmask, om_, lm_
        # window / shifted-window attention on the SD 512^2 latent grid (64 x 64 tokens)
        ww = workloads.make_inputs("sd_self", device=device)
        wB, wH, wN, _, wD = ww["shape"]
        win = {}
        for (wh, wwid, sh) in ((8, 8, 0), (8, 8, 4), (16, 16, 8)):
            msw = time_call(lambda: fa.fwd_window(ww["q"], ww["k"], ww["v"], 64, 64, wh, wwid, sh,
                                                  sh, scale=ww["scale"], stream=stream), 20)
            wfl = 4.0 * wB * wH * wN * (wh * wwid) * wD
            win[f"{wh}x{wwid}_shift{sh}"] = {"ms_per_step": round(msw, 4),
                                            "tflops": round(wfl / msw / 1e9, 1)}
        ext["window"] = {"workload": "sd_self grid 64x64, B2 H8 D64",
                         "note": "one attention launch that gathers and scatters the window "
                                 "rows itself; outputs allocated by the binding", "configs": win}
        del ww
        # causal at the benchmark shape: the useful FLOPs count keys j <= i only
        oc_, lc_ = torch.empty_like(q), torch.empty_like(lse)
        msc = time_call(lambda: fa.fa_fwd_ex(q, k, v, oc_, lc_, causal=True, scale=inp["scale"],
                                             stream=stream), max(5, args.steps // 10))
        kept = (Nq * (Nq + 1) // 2 if Nq <= Nk          # sum over rows i of min(i + 1, Nk)
                else Nk * (Nk + 1) // 2 + (Nq - Nk) * Nk)
        cfl = 4.0 * B * H * D * kept
        ext["causal"] = {"workload": args.workload, "ms_per_step": round(msc, 4),
                         "tflops_useful": round(cfl / msc / 1e9, 1),
                         "note": "FLOPs of the unmasked (j <= i) pairs only"}
        del oc_, lc_
        also["masks_causal_window"] = ext

    # ---- FP8 (e4m3 Q K^T) forward on the same workload, pre-pass included ----
    if args.also and rank == 0:
        ws8 = torch.empty(fa.fp8_workspace_bytes(B, H, Nq, Nk, D), dtype=torch.uint8, device=device)
        call8 = lambda: fa.fa_fwd_fp8(q, k, v, mask, out, lse, ws8, scale=inp["scale"], stream=stream)
        for _ in range(3):
            call8()
        torch.cuda.synchronize(device)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n8 = max(5, args.steps // 10)
        f0.record(stream)
        for _ in range(n8):
            call8()
        f1.record(stream)
        torch.cuda.synchronize(device)
        ms8 = f0.elapsed_time(f1) / n8
        also["fp8_qk"] = {"workload": args.workload, "ms_per_step": round(ms8, 4),
                          "tflops": round(flops / ms8 / 1e9, 1), "steps": n8,
                          "speedup_vs_bf16": round(ms_per_step / ms8, 3),
                          "note": "e4m3 Q K^T with K mean smoothing, bf16 P V; "
                                  "bf16-equivalent attention FLOPs; quantisation pre-pass timed"}
        del ws8

    # ---- split-key forward on a low-occupancy shape (2 units for all SMs) ----
    if args.also and rank == 0:
        sw = workloads.make_inputs("hunyuan_720p", device=device, B=1, H=2, Nq=256, Nk=119056)
        sB, sH, sNq, sNk, sD = sw["shape"]
        so = torch.empty_like(sw["q"])
        sl = torch.empty((sB, sH, sNq), dtype=torch.float32, device=device)
        sfl = accounting.attention_flops(sB, sH, sNq, sNk, sD)
        res = {"shape": f"B{sB} H{sH} Nq{sNq} Nk{sNk} D{sD}"}
        for tag, ranges in (("unsplit", 1), ("split", fa.split_count(sB, sH, sNq, sNk))):
            ws = torch.empty(max(16, fa.split_workspace_bytes(sB, sH, sNq, sD, ranges)),
                             dtype=torch.uint8, device=device)
            call = lambda: fa.fa_fwd_split(sw["q"], sw["k"], sw["v"], None, so, sl, ranges, ws,
                                           scale=sw["scale"], stream=stream)
            for _ in range(3):
                call()
            torch.cuda.synchronize(device)
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(20):
                call()
            a1.record(stream)
            torch.cuda.synchronize(device)
            sms = a0.elapsed_time(a1) / 20
            res[tag] = {"ranges": ranges, "ms_per_step": round(sms, 4),
                        "tflops": round(sfl / sms / 1e9, 1)}
        also["splitkv_long_keys"] = res
        del sw, so, sl

    peaks, peak_src = read_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    peak_sustained = peaks.get("bf16_tflops_sustained")

    # ---- secondary bound: one exponential per score on the MUFU pipe ----
    clock_summary = clocks.summary()
    ex2_rate = fa.measure_ex2_rate(stream)
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    clk_mhz = clock_summary.get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    exps = float(B) * H * Nq * Nk
    secondary = {"bound": "mufu_ex2", "ex2_per_clk_per_sm": round(ex2_rate, 2),
                 "sm_mhz": clk_mhz, "exp_bound_ms": round(exps / (ex2_rate * sm_count * clk_mhz * 1e6) * 1e3, 4),
                 "tensor_bound_ms": round(flops / (peak * 1e12) * 1e3, 4)}
    for v_ in also.values():
        if "tflops" in v_:
            v_["frac_of_peak"] = round(v_["tflops"] / peak, 4)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sampler = OracleSampler(inp)
        cflops, csecs, rows = sampler.run(sampler.rows_for(args.cpu_budget))
        cpu = {"value": cflops / csecs / 1e12, "unit": "TFLOP/s", "cores": sampler.threads,
               "kind": "oracle",
               "sample": f"{rows} seeded query rows per head x {B * H} heads of {args.workload} "
                         f"(all {Nk} keys), fp64 C oracle, {csecs:.1f} s",
               "extrapolated_full_s": round(csecs * Nq / rows, 1)}

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value_tflops, 2),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": args.workload + ("" if args.heads is None else f" (H {H})"),
                       "variant": variant, "B": B, "H": H, "Nq": Nq,
                       "Nk": Nk, "D": D,
                       "masked": mask is not None, "parallelism": f"replicas{world}",
                       "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB of Q/K/V per step)"},
            "pct_of_peak": round(100.0 * kernel_tflops / peak, 2),
            "step_ms": {"median": round(statistics.median(step_ms), 4),
                        "min": round(min(step_ms), 4), "max": round(max(step_ms), 4)},
            "clocks": clock_summary,
            "e2e": ({"value": round(e2e_tflops, 2), "unit": "TFLOP/s",
                     "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
                     "steps": e2e_steps, "h2d_gbs": round(h2d_gbs, 1),
                     "overlap": "double-buffered: upload i+1 (Q on one copy stream, K/V on "
                                "another) / download i-1 overlap kernel i"}
                    if e2e_steps else None),
            "gpu_launches": kernels_per_step * args.steps,
            "roofline": {"bound": "tensor", "achieved": round(kernel_tflops, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(kernel_tflops / peak, 4),
                         "traffic": read_traffic(args.workload),
                         "peak_source": f"{peak_src} bf16_tflops (burst; kernel timed alone)",
                         "frac_of_sustained": (round(kernel_tflops / float(peak_sustained), 4)
                                               if peak_sustained else None),
                         "secondary": secondary,
                         "algorithmic_flops_per_launch": flops,
                         "hbm_gbs": round(accounting.algorithmic_bytes(
                             B, H, Nq, Nk, D, masked=mask is not None) / (ms_per_step * 1e6), 1),
                         "algorithmic_bytes_per_launch": accounting.algorithmic_bytes(
                             B, H, Nq, Nk, D, masked=mask is not None)},
            "cpu_baseline": cpu,
        }
        if also:
            line["also"] = also
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bench_reference(args, world, rank, local):
    """The CPU oracle as it stands, on the machine's host cores, per step a bounded sample."""
    if rank != 0:
        return
    from unet_fa_fwd_gb300 import workloads

    w = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(w, device="cpu")
    B, H, Nq, Nk, D = inp["shape"]
    per_step = max(0.05, min(2.0, args.ref_budget / max(1, args.steps + args.warmup)))
    sampler = OracleSampler(inp)
    threads = sampler.threads
    nrows = sampler.rows_for(per_step)
    for _ in range(args.warmup):
        sampler.run(nrows)
    tot_f, tot_s, rows = 0.0, 0.0, nrows
    for _ in range(args.steps):
        f, s, rows = sampler.run(nrows)
        tot_f += f
        tot_s += s
    value = tot_f / tot_s / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "H": H, "Nq": Nq, "Nk": Nk, "D": D,
                   "masked": inp["mask"] is not None, "parallelism": "cpu"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step {rows} seeded query rows per head x {B * H} heads "
                                   f"(all {Nk} keys), fp64 C oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="hunyuan_720p")
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the workload's head count (smaller cases for profiling)")
    ap.add_argument("--variant", default="fwd",
                    choices=["fwd", "fp8", "causal", "key_mask", "additive_mask", "bool_mask", "window"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=90.0, help="seconds of oracle work, reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-also", dest="also", action="store_false")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.gpus != world:
        if world == 1 and args.gpus > 1:
            ap.error("--gpus N > 1 runs under torchrun (one process per GPU)")
    if args.impl == "reference":
        bench_reference(args, world, rank, local)
    else:
        bench_native(args, world, rank, local)


if __name__ == "__main__":
    main()
