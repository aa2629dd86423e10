#!/usr/bin/env python
"""Benchmark: attention fwd+bwd TFLOP/s on GB300 (and % of dense bf16 peak).

One step = one pass of the whole hot path over one batch of synthetic input:
forward (O, LSE), then the backward's D-vector preprocess, dK/dV kernel and dQ
kernel, all through the library's C ABI. The default workload is
B=4, Hq=32, Hkv=8, Tq=Tkv=4096, D=128, bf16, causal (seeded N(0,1) inputs).

FLOPs are counted by the headline convention: 4*B*Hq*Tq*Tkv*D for the
forward, 2.5x that for the backward, both halved under causal masking.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) every rank runs the same
workload on its own GPU (weak scaling, no collective on the data path); the
time is the max over ranks and the value the work of all ranks over it.
``--impl reference`` times the CPU double-precision oracle instead (rank 0
only), on a bounded sample of the same workload, extrapolated per step.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import fa_inputs  # noqa: E402

NOMINAL_BF16_TFLOPS = 2250.0
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------------ workload
def visible_pairs_per_head(w, rows=None) -> int:
    """(query, key) pairs the mask lets through in one head (optionally only
    for the query rows in ``rows``)."""
    lo, hi = (0, w.Tq) if rows is None else rows
    tot = 0
    for i in range(lo, hi):
        kh = min(w.Tkv, i + 1) if w.causal else w.Tkv
        kl = max(0, i - w.window + 1) if w.window > 0 else 0
        if w.window > 0 and not w.causal:
            tot += w.Tkv - min(kl, w.Tkv)   # the window hides past keys only
        else:
            tot += max(0, kh - kl)
    return tot


def counted_flops(w) -> tuple[float, float]:
    f = 4.0 * w.B * w.Hq * w.Tq * w.Tkv * w.D
    if w.causal:
        f *= 0.5
    return f, 2.5 * f


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"bf16_tflops": p.get("bf16_tflops"), "bf16_tflops_sustained": p.get("bf16_tflops_sustained"),
                "hbm_gbs": p.get("hbm_gbs"), "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


L2_NOTE = ("GPU arm: a 256 MiB buffer is written between timed steps (outside the step's "
           "events), and the step's working set exceeds the 126 MiB L2")

# A timed region at least this long runs the GPU under its power cap: the
# roofline then uses the sustained bf16 peak, otherwise the burst peak.
SUSTAINED_REGION_S = 2.0


def workload_config(w) -> dict:
    """The JSON line's config: the workload and the L2 rule, the same for both
    arms (how many GPUs run it is the line's n_gpus / parallelism)."""
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Tq": w.Tq, "Tkv": w.Tkv,
            "D": w.D, "causal": w.causal, "window": w.window, "seed": w.seed,
            "inputs": "seeded N(0,1), rounded to dtype", "l2": L2_NOTE}


def roofline_peak(peaks: dict, region_s: float) -> tuple[float, str]:
    """The bf16 peak a tensor-bound kernel is measured against: the sustained
    figure when the timed region lasts SUSTAINED_REGION_S or more (the clocks
    settle under the power cap), the burst figure for a shorter region."""
    if region_s >= SUSTAINED_REGION_S and peaks.get("bf16_tflops_sustained"):
        return peaks["bf16_tflops_sustained"], (
            f"{peaks['source']} sustained bf16 (timed region {region_s:.2f} s >= "
            f"{SUSTAINED_REGION_S:.0f} s)")
    return peaks["bf16_tflops"], (
        f"{peaks['source']} burst bf16 (timed region {region_s:.2f} s < "
        f"{SUSTAINED_REGION_S:.0f} s)")


KERNEL_SOURCES = {
    "fa_fwd_kernel": ["fa_fwd.cuh"],
    "fa_fwd_decode_kernel": ["fa_decode.cuh"],
    "fa_bwd_dq_decode_kernel": ["fa_decode.cuh"],
    "fa_bwd_dvec_kernel": ["fa_bwd.cuh"],
    "fa_bwd_dkv_kernel": ["fa_bwd_pipelined.cuh"],
    "fa_bwd_dkv_pair_kernel": ["fa_bwd_d256.cuh", "fa_bwd_pipelined.cuh"],
    "fa_bwd_dq_kernel": ["fa_bwd_pipelined.cuh"],
}
COMMON_SOURCES = ["fa_common.cuh", "sm103_ptx.cuh", "fa_inst.cuh", "fa_inst_d64.cu",
                  "fa_inst_d96.cu", "fa_inst_d128.cu", "fa_inst_d256.cu"]


def _code_only(text: str) -> str:
    """C++ source without comments, runs of whitespace collapsed (string
    literals in these sources hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_digest(kernel: str) -> str:
    """Digest of the code that defines ``kernel`` (its body, the shared device
    helpers and the tile configurations), comments and layout excluded."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_fa_fwd_03_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel] + COMMON_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as fh:
            h.update(name.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh)
    for r in rec.get("kernels", []):
        if (r.get("kernel") == kernel and r.get("workload") == workload
                and r.get("source_digest") == kernel_digest(kernel)):
            return r.get("dram_bytes_per_launch")
    return None


# ------------------------------------------------------------- multi-rank
def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest ``value`` over all ranks: a replicated job takes as long as
    its slowest rank. Uses the default process group when ``world > 1``."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, steps: int, flops_per_step: float, max_total_ms: float) -> float:
    """Whole-job TFLOP/s: each of ``world`` ranks runs ``steps`` full steps
    (weak scaling), timed by the slowest rank."""
    return world * steps * flops_per_step / (max_total_ms / 1e3) / 1e12


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of the SM clock and the throttle
    reasons; only the samples taken inside [t0, t1] (wall clock) count."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    @staticmethod
    def parse(out: str, t0: float, t1: float) -> dict:
        import datetime
        rows = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        nearest = False
        if not inside:
            # a region shorter than the sampling interval: the samples just
            # before and after it (within 0.1 s), marked as such
            before = [r for r in rows if t0 - 0.1 <= r[0] < t0][-1:]
            after = [r for r in rows if t1 < r[0] <= t1 + 0.1][:1]
            inside, nearest = before + after, True
        if not inside:
            return {"error": "no clock sample inside the timed region",
                    "samples_outside": len(rows)}
        sm = [r[1] for r in inside]
        mx = [r[2] for r in inside]
        pw, reasons = [], set()
        for r in inside:
            parts = r[3]
            try:
                pw.append(float(parts[4]))
            except ValueError:
                pass
            for name, val in zip(ClockSampler.NAMES, parts[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        r = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "sm_min_mhz": min(sm),
             "samples": len(sm), "reasons": sorted(reasons)}
        if nearest:
            r["nearest_samples"] = "region shorter than the 50 ms sampling interval"
        if pw:
            r["power_w_median"] = statistics.median(pw)
        return r

    def stop(self, *windows: tuple[float, float]) -> list[dict]:
        """Ends the sampling; one summary per (t0, t1) window."""
        if self.proc is None:
            return [{"error": "nvidia-smi unavailable"} for _ in windows]
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return [self.parse(out, t0, t1) for t0, t1 in windows]


def physical_gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x for x in vis.split(",") if x.strip()]
        if local_rank < len(ids) and ids[local_rank].strip().isdigit():
            return int(ids[local_rank])
    return local_rank


# ------------------------------------------------------------ CPU baseline
class OracleSample:
    """The oracle (fwd + bwd) on one (batch, KV group) slice of the workload:
    all its query heads, query rows [Tq - R, Tq) with R sized to take about a
    target time; the time per full step is extrapolated by visible pairs. The
    slice's inputs are generated once (the same seeded bits as the GPU run)."""

    def __init__(self, w):
        import oracle
        self.oracle = oracle
        self.w = w
        self.reps = w.Hq // w.Hkv
        x = fa_inputs.make_inputs(w)
        xs = [x["q"][0:1, 0:self.reps], x["k"][0:1, 0:1], x["v"][0:1, 0:1], x["do"][0:1, 0:self.reps]]
        self.xs = [t.double().numpy() for t in xs]
        self.total_pairs = w.B * w.Hq * visible_pairs_per_head(w)
        self.per_pair = None

    def run(self, rows):
        w = self.w
        lo = w.Tq - rows
        t0 = time.perf_counter()
        self.oracle.attn_fwd(*self.xs[:3], w.scale, w.causal, w.window, row_lo=lo, row_hi=w.Tq)
        self.oracle.attn_bwd(*self.xs, w.scale, w.causal, w.window, row_lo=lo, row_hi=w.Tq)
        return time.perf_counter() - t0, self.reps * visible_pairs_per_head(w, (lo, w.Tq))

    def rows_for(self, target_s: float) -> int:
        w = self.w
        if self.per_pair is None:
            dt, pairs = self.run(min(w.Tq, 8))
            self.per_pair = dt / max(pairs, 1)
        want_pairs = target_s / self.per_pair
        rows = min(w.Tq, 8)
        while rows < w.Tq and self.reps * visible_pairs_per_head(w, (w.Tq - rows, w.Tq)) < want_pairs:
            rows *= 2
        return min(rows, w.Tq)

    def step(self, target_s: float):
        """(seconds per full step, seconds spent, description)."""
        rows = self.rows_for(target_s)
        dt, pairs = self.run(rows)
        per_step = dt * self.total_pairs / pairs
        desc = (f"one (batch, KV group) slice ({self.reps} of {self.w.B * self.w.Hq} query heads), "
                f"query rows [{self.w.Tq - rows}, {self.w.Tq}): {pairs} of {self.total_pairs} visible "
                f"pairs, fwd + bwd in {dt:.2f} s, extrapolated by visible pairs")
        return per_step, dt, desc


def oracle_sample(w, target_s: float):
    """Time the oracle on a bounded sample of the workload (OracleSample):
    (seconds per full step, cores, description, seconds spent)."""
    smp = OracleSample(w)
    per_step, dt, desc = smp.step(target_s)
    return per_step, smp.oracle.num_threads(), desc, dt


# ---------------------------------------------------------------- our path
def host_link(hosts, outs, dev_bufs, s_in, s_out, reps: int = 3) -> dict:
    """Host <-> device copy rates of one step's tensors over pinned buffers:
    inputs in alone, outputs out alone, and both directions at once (ms per
    step's worth of bytes; GB/s)."""
    import torch

    def timed(copy_in: bool, copy_out: bool) -> float:
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_in)
            s_out.wait_event(e0)
            if copy_in:
                with torch.cuda.stream(s_in):
                    for n, t in hosts.items():
                        dev_bufs[n].copy_(t, non_blocking=True)
            if copy_out:
                with torch.cuda.stream(s_out):
                    for n, t in outs.items():
                        t.copy_(dev_bufs[n], non_blocking=True)
            s_in.wait_stream(s_out)
            e1.record(s_in)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return best

    bi = sum(t.numel() * t.element_size() for t in hosts.values())
    bo = sum(t.numel() * t.element_size() for t in outs.values())
    t_in, t_out, t_both = timed(True, False), timed(False, True), timed(True, True)
    return {"h2d_ms": round(t_in, 4), "h2d_gbs": round(bi / t_in / 1e6, 1),
            "d2h_ms": round(t_out, 4), "d2h_gbs": round(bo / t_out / 1e6, 1),
            "both_ms": round(t_both, 4), "both_gbs": round((bi + bo) / t_both / 1e6, 1)}


def run_ours(args, rank, world, local_rank):
    import torch
    import attention_fa_fwd_03_gb300 as fa

    w = fa_inputs.WORKLOADS[args.workload]
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    x = fa_inputs.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.Hq, w.Tq), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sc, ca, wi = w.scale, w.causal, w.window
    n_dkv = 1  # one dK/dV launch per step

    # A step as a user runs it: the forward and the backward through the public
    # API, each kernel launched while the previous one finishes (and dQ beside
    # dK/dV on masked grids); events only at the step's ends.
    def step_api(ev):
        ev[0].record()
        fa.fa_fwd(q, k, v, o, lse, sc, ca, wi)
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, sc, ca, wi, workspace=ws)
        ev[1].record()

    # The same step as its four phase calls with an event between each: the
    # events serialise the launches, so each pair brackets one kernel alone.
    def step_phases(ev):
        ev[0].record()
        fa.fa_fwd(q, k, v, o, lse, sc, ca, wi)
        ev[1].record()
        fa.fa_bwd_preprocess(o, do, ws)
        ev[2].record()
        fa.fa_bwd_dkv(q, k, v, do, lse, ws, dk, dv, sc, ca, wi)
        ev[3].record()
        fa.fa_bwd_dq(q, k, v, do, lse, ws, dq, sc, ca, wi)
        ev[4].record()

    def new_events(n):
        return [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    for _ in range(args.warmup):
        for fn, n in ((step_api, 2), (step_phases, 5)):
            flush.zero_()
            fn(new_events(n))
    torch.cuda.synchronize()
    if fa.fa_device_status() != 0:
        raise RuntimeError("a bounded device wait gave up during warm-up")

    def region(fn, n, steps):
        evs = [new_events(n) for _ in range(steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0, w0 = time.time(), time.perf_counter()
        for i in range(steps):
            flush.zero_()              # untimed: outside the step's event pair
            fn(evs[i])
        torch.cuda.synchronize()
        return evs, time.perf_counter() - w0, (t0, time.time())

    sampler = ClockSampler(physical_gpu_index(local_rank))
    sampler.start()
    # Each region starts after a short idle: measured, the first region after
    # one runs 3-5% faster than one that follows another region directly
    # (same sampled clock), so neither region inherits the other's load.
    time.sleep(0.25)
    # the timed region: the step through the public API (the line's value)
    evs, wall, win = region(step_api, 2, args.steps)
    time.sleep(0.25)
    # the per-kernel region, short (at most 100 steps, so its kernels run at
    # the clock of a burst, as the burst peak was measured): the same step as
    # phase calls (kernel times, roofline)
    kernel_steps = min(args.steps, 100)
    pevs, pwall, pwin = region(step_phases, 5, kernel_steps)
    if world > 1:
        torch.distributed.barrier()
    clocks, kernel_clocks = sampler.stop(win, pwin)
    status = fa.fa_device_status()

    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    phase_ms = [[e[j].elapsed_time(e[j + 1]) for e in pevs] for j in range(4)]
    phase_step_ms = [e[0].elapsed_time(e[4]) for e in pevs]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    fwd_f, bwd_f = counted_flops(w)
    value = job_tflops(world, args.steps, fwd_f + bwd_f, total_ms)

    # ---- end to end through the public API with host buffers
    e2e = None
    if rank == 0 or world > 1:
        hosts = {n: x[n].pin_memory() for n in ("q", "k", "v", "do")}
        outs = {"o": torch.empty_like(o, device="cpu").pin_memory(),
                "lse": torch.empty_like(lse, device="cpu").pin_memory(),
                "dq": torch.empty_like(dq, device="cpu").pin_memory(),
                "dk": torch.empty_like(dk, device="cpu").pin_memory(),
                "dv": torch.empty_like(dv, device="cpu").pin_memory()}
        h2d = sum(t.numel() * t.element_size() for t in hosts.values())
        d2h = sum(t.numel() * t.element_size() for t in outs.values())
        n_e2e = max(3, min(args.steps, args.e2e_steps))
        # A pipelined step loop, as a training input pipeline runs it: two sets
        # of device buffers; step i's inputs are copied in on one stream while
        # step i-1 computes on another and step i-2's results are copied out on
        # a third (events order each buffer set's copy-in, compute and copy-out).
        # Every step's copies are inside the timed region, from the first
        # step's copy-in to the last step's copy-out.
        s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        bufs = [{"q": q, "k": k, "v": v, "do": do, "o": o, "lse": lse, "dq": dq, "dk": dk,
                 "dv": dv, "ws": ws}]
        bufs.append({n: torch.empty_like(t) for n, t in bufs[0].items()})
        in_done = [torch.cuda.Event() for _ in range(2)]
        cmp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(i):
            j = i % 2
            bf = bufs[j]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(cmp_done[j])  # step i-2 is done reading this set
                for n in ("q", "k", "v", "do"):
                    bf[n].copy_(hosts[n], non_blocking=True)
                in_done[j].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_done[j])
                if i >= 2:
                    s_cmp.wait_event(out_done[j])  # step i-2's results are copied out
                fa.fa_fwd(bf["q"], bf["k"], bf["v"], bf["o"], bf["lse"], sc, ca, wi, stream=s_cmp)
                fa.fa_bwd(bf["q"], bf["k"], bf["v"], bf["o"], bf["do"], bf["lse"], bf["dq"],
                          bf["dk"], bf["dv"], sc, ca, wi, workspace=bf["ws"], stream=s_cmp)
                cmp_done[j].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[j])
                for n in ("o", "lse", "dq", "dk", "dv"):
                    outs[n].copy_(bf[n], non_blocking=True)
                out_done[j].record(s_out)

        for i in range(2):  # warm-up of both buffer sets
            e2e_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        s_cmp.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(n_e2e):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)
        link = host_link(hosts, outs, bufs[0], s_in, s_out)
        e2e = {"value": round(job_tflops(world, 1, fwd_f + bwd_f, e2e_ms), 2),
               "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 4),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "api": "fa_fwd + fa_bwd (C ABI via the Python binding), pinned host buffers; "
                      "copy-in, compute and copy-out on three streams over two buffer sets, "
                      "so step i's inputs load while step i-1 computes",
               "link": link,
               "bound_ms": round(max(link["both_ms"], sum(step_ms) / len(step_ms)), 4),
               "bound_note": "an end-to-end step takes at least the longer of the step's "
                             "copies in both directions at once and its compute"}

    if rank != 0:
        return None

    # ---- roofline of the dominant kernel
    peaks = load_peaks()
    pairs = w.B * w.Hq * visible_pairs_per_head(w)
    # query blocks of at most 8 rows per head run the split-key CUDA-core
    # forward and dQ kernels (latency- and HBM-bound: reported against HBM)
    short = w.Tq <= 8
    # head dim 256: dK/dV on two-CTA clusters
    names = ["fa_fwd_decode_kernel" if short else "fa_fwd_kernel", "fa_bwd_dvec_kernel",
             "fa_bwd_dkv_pair_kernel" if w.D == 256 else "fa_bwd_dkv_kernel",
             "fa_bwd_dq_decode_kernel" if short else "fa_bwd_dq_kernel"]
    avg_ms = [sum(p) / len(p) for p in phase_ms]
    # algorithmic work per launch: tensor FLOPs of each kernel's contractions over
    # the visible pairs (2*D per pair per contraction); bytes for the D-vector
    # pass and the split-key kernels (K and V read once per query head, the
    # head's query rows read and its output rows written)
    row_bytes = w.B * w.Hq * w.Tq * w.D * 2
    kv_bytes = w.B * w.Hq * w.Tkv * w.D * 2 * 2
    alg = {"fa_fwd_kernel": ("tensor", 2 * 2 * w.D * pairs),
           "fa_fwd_decode_kernel": ("hbm", kv_bytes + 2 * row_bytes + w.B * w.Hq * w.Tq * 4),
           "fa_bwd_dvec_kernel": ("hbm", 2 * w.B * w.Hq * w.Tq * w.D * 2 + w.B * w.Hq * w.Tq * 4),
           "fa_bwd_dkv_kernel": ("tensor", 4 * 2 * w.D * pairs),
           "fa_bwd_dkv_pair_kernel": ("tensor", 4 * 2 * w.D * pairs),
           "fa_bwd_dq_kernel": ("tensor", 3 * 2 * w.D * pairs),
           "fa_bwd_dq_decode_kernel": ("hbm", kv_bytes + 3 * row_bytes + 2 * w.B * w.Hq * w.Tq * 4)}
    kernels = {}
    for nm, ms in zip(names, avg_ms):
        bound, work = alg[nm]
        if bound == "tensor":
            kernels[nm] = {"ms": round(ms, 4), "tflops": round(work / (ms / 1e3) / 1e12, 2)}
        else:
            kernels[nm] = {"ms": round(ms, 4), "gbs": round(work / (ms / 1e3) / 1e9, 1)}
    dom = names[max(range(4), key=lambda j: avg_ms[j])]
    bound, work = alg[dom]
    launches = n_dkv if dom in ("fa_bwd_dkv_kernel", "fa_bwd_dkv_pair_kernel") else 1
    launch_s = avg_ms[names.index(dom)] / launches / 1e3
    work_per_launch = work / launches
    region_s = sum(phase_step_ms) / 1e3  # the region the kernel times come from
    if bound == "tensor":
        achieved = work_per_launch / launch_s / 1e12
        peak, peak_source = roofline_peak(peaks, region_s)
        unit = "TFLOP/s"
    else:
        achieved = work_per_launch / launch_s / 1e9
        peak, peak_source = peaks["hbm_gbs"], f"{peaks['source']} HBM copy"
        unit = "GB/s"
    traffic = ncu_traffic(dom, w.name)
    roofline = {"kernel": dom, "bound": bound, "achieved": round(achieved, 2), "peak": peak,
                "unit": unit, "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": peak_source,
                "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4) if bound == "tensor" else None,
                "frac_of_sustained": (round(achieved / peaks["bf16_tflops_sustained"], 4)
                                      if bound == "tensor" else None),
                "work_per_launch": work_per_launch,
                "work_definition": "tensor FLOPs of the kernel's own contractions over the visible "
                                   "(query, key) pairs: 2*D per pair per contraction (fwd 2, dK/dV 4, dQ 3)"}

    cpu = None
    if not args.no_cpu_baseline:
        per_step_s, cores, desc, took = oracle_sample(w, args.cpu_seconds)
        cpu = {"value": round((fwd_f + bwd_f) / per_step_s / 1e12, 6), "unit": "TFLOP/s",
               "cores": cores, "kind": "oracle", "sample": desc,
               "seconds_per_full_step": round(per_step_s, 1)}

    ms_step = total_ms / args.steps
    fwd_ms = sum(phase_ms[0]) / kernel_steps
    bwd_ms = sum(sum(p) for p in phase_ms[1:]) / kernel_steps
    line = {
        "metric": "attention fwd+bwd TFLOP/s at 1 GB300 (and % of dense bf16 peak)",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w),
        "parallelism": f"replicas x{world} (each GPU runs the full workload, no collective)",
        "pct_of_nominal_bf16_peak": round(100 * value / world / NOMINAL_BF16_TFLOPS, 2),
        "pct_of_measured_bf16_peak": round(100 * value / world / peaks["bf16_tflops"], 2),
        "fwd_tflops": round(fwd_f / (fwd_ms / 1e3) / 1e12, 2),
        "bwd_tflops": round(bwd_f / (bwd_ms / 1e3) / 1e12, 2),
        "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4),
        "step_calls": "fa_fwd + fa_bwd through the public API, events at the step's ends only",
        "phase_ms_per_step": round(sum(phase_step_ms) / kernel_steps, 4),
        "kernels": kernels,
        "kernels_region": {"steps": kernel_steps, "clocks": kernel_clocks,
                           "what": ("the same step as the four phase calls with an event between "
                                    "launches (which serialises them), after the timed region and "
                                    "a 0.25 s idle; fwd_ms, bwd_ms, kernels and the roofline come "
                                    "from it")},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (3 + n_dkv),
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
        "wall_s_kernels_region": round(pwall, 4),
        "device_status": status,
    }
    return line


# ----------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle as the reference arm: each of warm-up + timed steps runs a
    bounded sample of the workload (sized so the whole run takes about two
    minutes), extrapolated to a full step."""
    w = fa_inputs.WORKLOADS[args.workload]
    fwd_f, bwd_f = counted_flops(w)
    smp = OracleSample(w)
    budget = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    per_step = []
    desc = None
    for i in range(args.warmup + args.steps):
        s, _, desc = smp.step(budget)
        if i >= args.warmup:
            per_step.append(s)
    mean_s = sum(per_step) / len(per_step)
    value = (fwd_f + bwd_f) / mean_s / 1e12
    cores = smp.oracle.num_threads()
    return {
        "metric": "attention fwd+bwd TFLOP/s at 1 GB300 (and % of dense bf16 peak)",
        "impl": "reference", "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_s * 1e3, 1),
        "ms_per_step_extrapolated": True,
        "ms_per_step_method": ("each step times the oracle on a bounded sample (a query-row range "
                               "of one (batch, KV group) slice) and scales it to the full workload "
                               "by visible (query, key) pairs; not a measured full step"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=fa_inputs.HEADLINE, choices=sorted(fa_inputs.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    try:
        line = run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
