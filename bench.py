#!/usr/bin/env python3
"""Benchmark of the skinny decode projection on one GB300 (or N replicas).

Metric: weight-stream GB/s (and us per projection) against the HBM roofline,
at decode batch M = 1..64.  One step = one pass of the whole hot path over
one batch of synthetic inputs:

  sweep (default)  the batch sweep M in {1,2,4,8,16,32,64}, K = N = 7168,
                   bf16, no residual: 7 projections, each with its own
                   102.8 MB weight (seed = index of M), so a step streams
                   719 MB of weights and no weight is L2-resident when its
                   projection runs (inputs larger than the 126 MB L2).
  chain            the five projections of a decode layer at M = 1, 8, 64.
  wide / deepk     the wide input projection and the deep-K output projection
                   with residual, at their M values.
  pr1              the single M = 1, K = N = 1024 projection with residual.

The headline `value` is the whole job's weight bytes / device time of exactly
`--steps` eager steps (CUDA events only at the two ends of the timed region,
max over ranks).  Every other figure comes from separate passes after it, so
no event sits between two launches of the timed region (an event between two
launches ends their programmatic overlap):

  per_projection   for every projection of the step, `us_back_to_back`: a run
                   of launches of that projection alone, each over a different
                   copy of its weight (the copies together exceed twice the
                   L2), events at the two ends of the run, time / launches;
                   `us_event_isolated`: events before and after each launch in
                   sampled steps.
  roofline         the dominant kernel (most device time in the step): its
                   projections' algorithmic bytes summed / their
                   back-to-back times summed, against the measured HBM peak.
  kernel_in_step   each kernel kind's consecutive launches inside sampled
                   steps, events at the kind boundaries only.
  configs          the other named workloads (wide, deep-K, PR1, the chain
                   with and without the L2 prefetch of the next weight) with
                   the same fields, unless --headline-only.

`e2e` repeats the headline measurement through the public API with the
step's activations copied from pinned host memory and its outputs copied
back inside the timed region (weights stay resident: they are parameters,
not per-step inputs).  `--impl reference` times the CPU oracle on the same
metric instead (a bounded sample of each step).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "weight-stream GB/s and µs/projection vs GB300 HBM roofline at M=1..64"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
EXTRA_CONFIGS = ("wide", "deepk", "pr1", "chain")


# ------------------------------------------------------------------ workloads
def workload(name: str):
    from projection_gemm_gb300 import inputs as I
    if name == "sweep":
        projs = [I.sweep(m) for m in I.SWEEP_M]
        desc = ("batch sweep M in {1,2,4,8,16,32,64}, K=N=7168, bf16 W~N(0,1/K), x~N(0,1), "
                "no residual, seed = index of M")
        return projs, desc, {"M": list(I.SWEEP_M), "N": 7168, "K": 7168, "epilogue": "bf16"}
    if name == "wide":
        return ([I.wide(m) for m in I.WIDE_M], "wide input projection M in {1,2,8,32,64}, K=7168, N=12288, "
                "1% of W rows x16", {"M": list(I.WIDE_M), "N": 12288, "K": 7168, "epilogue": "bf16"})
    if name == "deepk":
        return ([I.deepk(m) for m in I.DEEPK_M], "deep-K output projection + residual M in {1,4,16,64}, "
                "K=16384, N=7168, residual~N(0,4)", {"M": list(I.DEEPK_M), "N": 7168, "K": 16384,
                                                     "epilogue": "bf16_residual"})
    if name == "chain":
        projs = [p for m in I.CHAIN_M for p in I.chain(m)]
        return projs, ("decode-layer chain at M in {1,8,64}: 7168->12288, 8192->7168 (+res), "
                       "7168->384 (fp32), 7168->4096, 4096->7168 (+res)"), \
            {"M": list(I.CHAIN_M), "stages": [list(s) for s in I.CHAIN_STAGES]}
    if name == "pr1":
        return [I.pr1()], "PR1: M=1, K=N=1024, + residual", {"M": [1], "N": 1024, "K": 1024,
                                                              "epilogue": "bf16_residual"}
    raise ValueError(name)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash(kernel: str) -> str:
    """sha256 of the CUDA source that defines `kernel` (its ncu counters are
    only valid for that exact source)."""
    import hashlib
    srcs = {"splitk_tc": ("skg_splitk_tc.cu", "skg_tc_common.cuh"), "gemv": ("skg_gemv.cu",)}.get(kernel)
    if srcs is None:
        return ""
    h = hashlib.sha256()
    for src in srcs:
        with open(os.path.join(ROOT, "projection_gemm_gb300", "csrc", src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu record, or None when the
    record is missing or was taken on a different version of the kernel."""
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.txt")
    try:
        rec = json.load(open(path))
    except Exception:
        return None
    if rec.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return rec.get("bytes_per_launch")


# --------------------------------------------------------------- clock probe
class ClockSampler:
    """nvidia-smi samples (every 100 ms) while the GPU passes run."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: str):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, windows):
        """Median SM clock and the reasons seen over the given (t0, t1)
        windows (each widened by one sampling period)."""
        rows = [s for t, s in self.samples if any(a - 0.1 <= t <= b + 0.1 for a, b in windows)]
        sm, mx, reasons, power = [], None, set(), []
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(self.NAMES, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "sm_mhz_min": min(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------ distributed
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def aggregate(elapsed_s: float, units: float, world: int):
    """Max of the elapsed time and sum of the units over all ranks."""
    if world == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------- CPU oracle
class OracleSample:
    """The oracle over the first R W rows of every projection of one step, R
    calibrated once for about `seconds` of CPU work (the oracle as it stands,
    all host cores through its OpenMP loop); when the whole step takes less
    than that, the whole step repeated."""

    def __init__(self, data, seconds: float):
        import oracle.oracle as O
        self.O = O
        self.data = data            # [(Projection, x bits, W bits, residual bits or None)]
        b, dt = self.run_rows(16)
        nmax = max(p.N for p, *_ in data)
        self.rows = max(16, min(nmax, int(16 * seconds / max(dt, 1e-6))))
        self.reps = 1
        if self.rows == nmax:
            _, dt_full = self.run_rows(nmax)
            self.reps = max(1, int(seconds / max(dt_full, 1e-6)))
        self.cores = O.max_threads()
        what = (f"the whole step ({len(data)} projections, every M, all W rows), {self.reps} times"
                if self.rows == nmax else
                f"the first {self.rows} W rows of each of the step's {len(data)} projections, every M")
        self.desc = f"oracle (fp64, {self.cores} threads) on {what}"

    def run_rows(self, rows):
        import numpy as np
        wbytes = 0
        t0 = time.perf_counter()
        for p, xb, wb, rb in self.data:
            r = min(rows, p.N)
            self.O.linear(xb, np.ascontiguousarray(wb[:r]),
                          None if rb is None else np.ascontiguousarray(rb[:, :r]))
            wbytes += 2 * r * p.K
        return wbytes, time.perf_counter() - t0

    def run(self):
        b = dt = 0.0
        for _ in range(self.reps):
            b1, dt1 = self.run_rows(self.rows)
            b, dt = b + b1, dt + dt1
        return b / dt / 1e9, dt


def host_data(projs):
    from projection_gemm_gb300.inputs import bits, generate
    out = []
    for p in projs:
        t = generate(p)
        out.append((p, bits(t.x), bits(t.W), None if t.res is None else bits(t.res)))
    return out


# ------------------------------------------------------------ device set-up
class DeviceWorkload:
    """One workload's operands resident in HBM and one plan per projection.

    A step's activations (x, residual) and its outputs each live in one
    packed buffer (256-byte aligned segments), so the end-to-end run moves
    them with one host->device and one device->host copy per step.  Launch
    arguments are kept as raw device addresses, so a launch costs the host
    one call into the library."""

    def __init__(self, name, dev, pdl=True, keep_host=False, host_bits=False):
        import torch

        from projection_gemm_gb300 import skg
        from projection_gemm_gb300.inputs import bits, generate
        self.name = name
        self.projs, self.desc, self.cfg = workload(name)
        gens = [generate(p) for p in self.projs]

        def seg(nbytes):
            return (nbytes + 255) // 256 * 256
        in_bytes = sum(seg(t.x.numel() * 2) + (seg(t.res.numel() * 2) if t.res is not None else 0) for t in gens)
        out_bytes = sum(seg(p.M * p.N * p.out_bytes_per_elem) for p in self.projs)
        self.dev_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        self.dev_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        self.host_in = host_in if keep_host else None
        self.host_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory() if keep_host else None

        def view(buf, off, shape, dt):
            n = shape[0] * shape[1] * torch.empty((), dtype=dt).element_size()
            return buf[off:off + n].view(dt).view(*shape)

        self.ops, self.host = [], []
        self.in_segs, self.out_segs = [], []     # (offset, bytes) of each projection's inputs / output
        oi = oo = 0
        for p, t in zip(self.projs, gens):
            oi0, oo0 = oi, oo
            if host_bits:
                self.host.append((p, bits(t.x), bits(t.W), None if t.res is None else bits(t.res)))
            plan = skg.Plan(p.M, p.N, p.K, p.epilogue)
            plan.set_pdl(bool(pdl))
            dt = torch.float32 if p.epilogue == "fp32" else torch.bfloat16
            x = view(self.dev_in, oi, (p.M, p.K), torch.bfloat16)
            view(host_in, oi, (p.M, p.K), torch.bfloat16).copy_(t.x)
            oi += seg(t.x.numel() * 2)
            res = None
            if t.res is not None:
                res = view(self.dev_in, oi, (p.M, p.N), torch.bfloat16)
                view(host_in, oi, (p.M, p.N), torch.bfloat16).copy_(t.res)
                oi += seg(t.res.numel() * 2)
            y = view(self.dev_out, oo, (p.M, p.N), dt)
            oo += seg(p.M * p.N * p.out_bytes_per_elem)
            self.in_segs.append((oi0, oi - oi0))
            self.out_segs.append((oo0, oo - oo0))
            W = t.W.to(dev)
            self.ops.append(dict(p=p, plan=plan, info=plan.info(), x=x, W=W, res=res, y=y,
                                 args=(x.data_ptr(), W.data_ptr(), None if res is None else res.data_ptr(),
                                       y.data_ptr())))
        self.dev_in.copy_(host_in)
        del gens
        self.pools = None

    def weight_bytes(self):
        return sum(o["p"].weight_bytes() for o in self.ops)

    def e2e_step(self, main, cin, cout):
        """One step end to end, issued on torch streams (for capture as one
        graph): the first projection's inputs are copied from pinned host
        memory on `main` and the rest on `cin`, which `main` waits for
        before the second launch; each projection's output is copied back on
        `cout` as soon as its launch completes, so only the first input copy
        and the last output copy are not overlapped with a kernel."""
        import torch
        (a0, n0) = self.in_segs[0]
        cin.wait_stream(main)
        cout.wait_stream(main)
        self.dev_in[a0:a0 + n0].copy_(self.host_in[a0:a0 + n0], non_blocking=True)
        rest = None
        if len(self.ops) > 1:
            with torch.cuda.stream(cin):
                self.dev_in[a0 + n0:].copy_(self.host_in[a0 + n0:], non_blocking=True)
            rest = cin.record_event()
        for i, o in enumerate(self.ops):
            if i == 1:
                main.wait_event(rest)
            self.launch(o, main.cuda_stream)
            cout.wait_event(main.record_event())
            a, n = self.out_segs[i]
            with torch.cuda.stream(cout):
                self.host_out[a:a + n].copy_(self.dev_out[a:a + n], non_blocking=True)
        main.wait_stream(cout)

    def launch(self, o, s, W=None):
        from projection_gemm_gb300 import skg
        x, w, r, y = o["args"]
        skg.skg_run(o["plan"].handle, x, w if W is None else W, r, y, s)

    def step(self, s, events=None, at=None, side=None, side_join=True):
        """One pass over every projection on stream handle `s`.  events: a
        list of CUDA events recorded before the launches whose indices are in
        `at` (all launches when `at` is None) and after the last one.  side:
        (torch stream, its handle) on which each projection's successor gets
        its L2 prefetch (skg_prefetch_l2) issued beside it."""
        from projection_gemm_gb300 import skg
        j = 0
        n = len(self.ops)
        for i, o in enumerate(self.ops):
            if events is not None and (at is None or i in at):
                events[j].record(self._streams[s])
                j += 1
            if side is not None and i + 1 < n:
                if side_join:
                    side[0].wait_stream(self._streams[s])
                nx = self.ops[i + 1]
                skg.skg_prefetch_l2(nx["plan"].handle, nx["args"][1], side[1])
            self.launch(o, s)
            if side is not None and side_join and i + 1 < n:
                self._streams[s].wait_stream(side[0])
        if side is not None and not side_join:
            self._streams[s].wait_stream(side[0])
        if events is not None:
            events[j].record(self._streams[s])

    def bind_streams(self, streams):
        self._streams = {s.cuda_stream: s for s in streams}

    def weight_pools(self, l2_bytes):
        """Per (N, K): the workload's own weights of that shape, plus copies
        until they hold at least twice the L2 (at least two)."""
        if self.pools is None:
            pools = {}
            for o in self.ops:
                pools.setdefault((o["p"].N, o["p"].K), []).append(o["W"])
            for ws in pools.values():
                i = 0
                while len(ws) < 2 or sum(w.numel() * 2 for w in ws) < 2 * l2_bytes:
                    ws.append(ws[i].clone())
                    i += 1
            self.pools = {k: [w.data_ptr() for w in ws] for k, ws in pools.items()}
            self._pool_tensors = pools
        return self.pools

    def close(self):
        for o in self.ops:
            o["plan"].check()
            o["plan"].close()
        self.ops = []
        self.pools = None
        self._pool_tensors = None


def t_ideal_us(p, peak_hbm, peak_tf):
    return max(p.algorithmic_bytes() / (peak_hbm * 1e9), p.flops() / (peak_tf * 1e12)) * 1e6


def bar_for(p):
    """The acceptance bar on a projection's roofline fraction: 0.80 for
    M <= 16, 0.70 for M >= 32; PR1 (2 MB, below launch latency) has none."""
    if p.name == "pr1":
        return None
    return 0.80 if p.M <= 16 else 0.70


def measure_back_to_back(wl, s, torch_stream, l2_bytes, min_launches=28, reps=5):
    """us per launch of each projection, launched alone back to back over
    distinct weight copies.  The run is captured once as a CUDA graph (the
    programmatic launch edges are kept) so that the host's launch rate never
    limits it, and replayed `reps` times with events at its two ends."""
    import torch
    pools = wl.weight_pools(l2_bytes)
    cap = torch.cuda.Stream(device=torch_stream.device)
    out = []
    for o in wl.ops:
        pool = pools[(o["p"].N, o["p"].K)]
        seq = pool * max(1, -(-min_launches // len(pool)))
        cap.wait_stream(torch_stream)
        with torch.cuda.stream(cap):
            for w in seq:                           # eager once: first-use set-up outside the capture
                wl.launch(o, cap.cuda_stream, W=w)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for w in seq:
                wl.launch(o, cap.cuda_stream, W=w)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps + 1)]
        for a, b in evs:
            a.record(torch_stream)
            g.replay()
            b.record(torch_stream)
        torch.cuda.synchronize()
        t = [a.elapsed_time(b) * 1e3 / len(seq) for a, b in evs[1:]]
        out.append((statistics.median(t), len(seq) * reps))
        del g
    return out


def measure_event_isolated(wl, s, torch_stream, steps=24):
    """us of each launch with events right before and after it, in whole
    steps (median over the steps)."""
    import torch
    n = len(wl.ops)
    per = [[] for _ in range(n)]
    for _ in range(steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        wl.step(s, events=ev)
        torch.cuda.synchronize()
        for i in range(n):
            per[i].append(ev[i].elapsed_time(ev[i + 1]) * 1e3)
    return [statistics.median(v) for v in per]


def measure_kind_runs(wl, s, torch_stream, steps=24):
    """Each run of consecutive launches of one kernel kind inside whole
    steps, events at the kind boundaries only: us per step per kind."""
    import torch
    runs, a = [], 0
    for i in range(1, len(wl.ops) + 1):
        if i == len(wl.ops) or wl.ops[i]["info"]["kernel"] != wl.ops[a]["info"]["kernel"]:
            runs.append((a, i))
            a = i
    at = {r[0] for r in runs}
    tot = {}
    for _ in range(steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(runs) + 1)]
        wl.step(s, events=ev, at=at)
        torch.cuda.synchronize()
        for j, (a, b) in enumerate(runs):
            k = wl.ops[a]["info"]["kernel"]
            d = tot.setdefault(k, {"launches_per_step": 0, "us": []})
            d["us"].append(ev[j].elapsed_time(ev[j + 1]) * 1e3)
    for j, (a, b) in enumerate(runs):
        k = wl.ops[a]["info"]["kernel"]
        tot[k].setdefault("bytes_per_step", 0)
        tot[k]["bytes_per_step"] += sum(wl.ops[i]["p"].algorithmic_bytes() for i in range(a, b))
        tot[k]["launches_per_step"] += b - a
    out = {}
    for k, d in tot.items():
        # one sample per step per run of this kind: sum the runs of a step
        nr = sum(1 for a, b in runs if wl.ops[a]["info"]["kernel"] == k)
        per_step = [sum(d["us"][i:i + nr]) for i in range(0, len(d["us"]), nr)]
        us = statistics.median(per_step)
        out[k] = {"launches_per_step": d["launches_per_step"], "bytes_per_step": d["bytes_per_step"],
                  "us_per_step": round(us, 3), "gbs": round(d["bytes_per_step"] / us / 1e3, 1)}
    return out


def e2e_pipelined(wl, stream, steps, wbytes_step):
    """End to end with the copies overlapped: two sets of activation and
    output buffers, step k's input copy (copy stream) and output copy (a
    second copy stream) overlapping the kernels of steps k -/+ 1 (each set's
    launches captured as one CUDA graph); the host waits once, at the end."""
    import torch
    dev = stream.device
    sets = [(wl.dev_in, wl.dev_out)]
    sets.append((torch.empty_like(wl.dev_in), torch.empty_like(wl.dev_out)))
    sets[1][0].copy_(sets[0][0])
    host_out = [wl.host_out, torch.empty_like(wl.host_out).pin_memory()]
    graphs = []
    cap = torch.cuda.Stream(device=dev)
    for din, dout in sets:
        # the same launches, pointed at this set's buffers
        saved = [o["args"] for o in wl.ops]
        for o in wl.ops:
            x, w, r, y = o["args"]
            shift_in = din.data_ptr() - wl.dev_in.data_ptr()
            shift_out = dout.data_ptr() - wl.dev_out.data_ptr()
            o["args"] = (x + shift_in, w, None if r is None else r + shift_in, y + shift_out)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            wl.step(cap.cuda_stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            wl.step(cap.cuda_stream)
        torch.cuda.synchronize()
        graphs.append(g)
        for o, a in zip(wl.ops, saved):
            o["args"] = a
    cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {}

    def issue(k):
        j = k % 2
        din, dout = sets[j]
        if k >= 2:
            cin.wait_event(ev[("comp", k - 2)])          # set j's inputs are free again
        with torch.cuda.stream(cin):
            din.copy_(wl.host_in, non_blocking=True)
        ev[("in", k)] = cin.record_event()
        stream.wait_event(ev[("in", k)])
        if k >= 2:
            stream.wait_event(ev[("out", k - 2)])        # set j's outputs were copied back
        graphs[j].replay()
        ev[("comp", k)] = stream.record_event()
        cout.wait_event(ev[("comp", k)])
        with torch.cuda.stream(cout):
            host_out[j].copy_(dout, non_blocking=True)
        ev[("out", k)] = cout.record_event()
    for k in range(4):
        issue(k)
    torch.cuda.synchronize()
    ev.clear()
    t0 = time.perf_counter()
    for k in range(steps):
        issue(k)
    torch.cuda.synchronize()
    te = time.perf_counter() - t0
    del graphs
    return {"value": round(wbytes_step * steps / te / 1e9, 1), "unit": "GB/s", "steps": steps,
            "ms_per_step": round(te / steps * 1e3, 4),
            "how": ("two buffer sets; each step's input copy, kernels (one CUDA graph replay) and output copy "
                    "on three streams, ordered by events, so copies overlap the neighbouring steps' kernels; "
                    "the host waits once at the end")}


def timed_pass(wl, s, torch_stream, steps, **kw):
    """Device seconds of `steps` whole steps, events at the two ends only."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(torch_stream)
    for _ in range(steps):
        wl.step(s, **kw)
    b.record(torch_stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3


def projection_table(wl, b2b, iso, peak_hbm, peak_tf):
    out = {}
    for o, (us, launches), us_iso in zip(wl.ops, b2b, iso if iso else [None] * len(wl.ops)):
        p, info = o["p"], o["info"]
        ti = t_ideal_us(p, peak_hbm, peak_tf)
        row = {"M": p.M, "N": p.N, "K": p.K, "epilogue": p.epilogue, "kernel": info["kernel"],
               "split": info["split_k"], "grid": info["grid"], "stages": info["stages"],
               "algorithmic_bytes": p.algorithmic_bytes(), "t_ideal_us": round(ti, 3),
               "us_back_to_back": round(us, 3), "launches_timed": launches,
               "weight_gbs": round(p.weight_bytes() / us / 1e3, 1),
               "frac_back_to_back": round(ti / us, 4)}
        if us_iso is not None:
            row["us_event_isolated"] = round(us_iso, 3)
            row["frac_event_isolated"] = round(ti / us_iso, 4)
        bar = bar_for(p)
        if bar is not None:
            row["bar"] = bar
            row["meets_bar"] = bool(ti / us >= bar)
        out[p.name] = row
    return out


def roofline_from(table, wl, peak_hbm, peak_src, workload_name):
    """The dominant kernel of the step (largest summed back-to-back time):
    its projections' algorithmic bytes / their back-to-back time."""
    kinds = {}
    for o in wl.ops:
        r = table[o["p"].name]
        k = kinds.setdefault(r["kernel"], {"bytes": 0, "us": 0.0, "projections": []})
        k["bytes"] += r["algorithmic_bytes"]
        k["us"] += r["us_back_to_back"]
        k["projections"].append(o["p"].name)
    dom = max(kinds, key=lambda k: kinds[k]["us"])
    d = kinds[dom]
    achieved = d["bytes"] / (d["us"] * 1e-6) / 1e9
    return {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak_hbm, "unit": "GB/s",
            "frac": round(achieved / peak_hbm, 4), "traffic": kernel_traffic(dom, workload_name),
            "peak_source": (f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback"),
            "bytes_per_pass": d["bytes"], "us_per_pass": round(d["us"], 3), "projections": d["projections"],
            "timing": ("achieved = bytes_per_pass / us_per_pass: the sum of this kernel's projections' algorithmic "
                       "bytes over the sum of their us_back_to_back (per_projection), measured after the timed "
                       "region")}


def measure_config(name, dev, s, torch_stream, args, peak_hbm, peak_tf, l2_bytes, seconds=0.3):
    """A named workload besides the headline: whole-step GB/s of a short
    eager pass, and its per-projection figures."""
    wl = DeviceWorkload(name, dev, pdl=bool(args.pdl))
    wl.bind_streams([torch_stream])
    try:
        for _ in range(3):
            wl.step(s)
        t1 = timed_pass(wl, s, torch_stream, 1)
        steps = max(5, min(400, int(seconds / max(t1, 1e-6))))
        el = timed_pass(wl, s, torch_stream, steps)
        b2b = measure_back_to_back(wl, s, torch_stream, l2_bytes)
        iso = measure_event_isolated(wl, s, torch_stream, steps=12)
        table = projection_table(wl, b2b, iso, peak_hbm, peak_tf)
        out = {"workload": wl.desc, "steps": steps, "us_per_step": round(el / steps * 1e6, 3),
               "gbs": round(wl.weight_bytes() * steps / el / 1e9, 1), "per_projection": table}
        bars = [r for r in table.values() if "bar" in r]
        out["projections_meeting_bar"] = f"{sum(r['meets_bar'] for r in bars)}/{len(bars)}"
        if name == "chain":
            out["variants"] = chain_variants(wl, s, torch_stream, steps, l2_bytes)
        return out
    finally:
        wl.close()


def chain_graph(wl, torch_stream, steps, side_frac=None):
    """The chain's whole step captured once as a CUDA graph (programmatic
    edges between its launches) and replayed; with side_frac, each next
    weight's skg_prefetch_l2 runs on a forked side-stream branch of the graph,
    joined before the next projection."""
    import torch
    from projection_gemm_gb300 import skg
    dev = torch_stream.device
    cap, side = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    wl.bind_streams([cap, side])
    kw = {}
    if side_frac is not None:
        for o in wl.ops:
            skg.skg_plan_set_prefetch_fraction(o["plan"].handle, side_frac)
        kw = {"side": (side, side.cuda_stream), "side_join": True}
    cap.wait_stream(torch_stream)
    with torch.cuda.stream(cap):
        wl.step(cap.cuda_stream, **kw)        # descriptors and attributes outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        wl.step(cap.cuda_stream, **kw)
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    main = torch.cuda.current_stream(dev)      # replay() launches on the current stream
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(main)
    for _ in range(steps):
        g.replay()
    b.record(main)
    torch.cuda.synchronize()
    el = a.elapsed_time(b) / 1e3
    del g
    wl.bind_streams([torch_stream])
    return {"us_per_step": round(el / steps * 1e6, 3), "gbs": round(wl.weight_bytes() * steps / el / 1e9, 1)}


def chain_variants(wl, s, torch_stream, steps, l2_bytes):
    """The chain end to end per M and in total, without prefetch, with the
    in-launch prefetch of the next weight, and with skg_prefetch_l2 of the
    next weight on a side stream (joined before the next projection, as the
    pages' side stream is, and fire-and-forget with one join per step)."""
    import torch
    from projection_gemm_gb300 import inputs as I
    side = torch.cuda.Stream(device=torch_stream.device)
    wl.bind_streams([torch_stream, side])
    per_m = len(I.CHAIN_STAGES)
    seg_at = set(range(0, len(wl.ops), per_m))

    def set_next(frac):
        for i, o in enumerate(wl.ops):
            if frac > 0 and (i + 1) % per_m != 0:
                nx = wl.ops[i + 1]
                o["plan"].set_next_weight(nx["W"], int(min(nx["p"].weight_bytes(), frac * l2_bytes)))
            else:
                o["plan"].set_next_weight(None, 0)

    def one(label, frac=0.0, side_frac=None, join=True):
        set_next(frac)
        kw = {}
        if side_frac is not None:
            from projection_gemm_gb300 import skg
            for o in wl.ops:
                skg.skg_plan_set_prefetch_fraction(o["plan"].handle, side_frac)
            kw = {"side": (side, side.cuda_stream), "side_join": join}
        for _ in range(3):
            wl.step(s, **kw)
        el = timed_pass(wl, s, torch_stream, steps, **kw)
        # per M: events at the M boundaries only
        seg = [[] for _ in range(len(I.CHAIN_M))]
        for _ in range(12):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(I.CHAIN_M) + 1)]
            wl.step(s, events=ev, at=seg_at, **kw)
            torch.cuda.synchronize()
            for j in range(len(I.CHAIN_M)):
                seg[j].append(ev[j].elapsed_time(ev[j + 1]) * 1e3)
        res = {"us_per_step": round(el / steps * 1e6, 3), "gbs": round(wl.weight_bytes() * steps / el / 1e9, 1),
               "per_m": {}}
        for j, m in enumerate(I.CHAIN_M):
            us = statistics.median(seg[j])
            wb = sum(o["p"].weight_bytes() for o in wl.ops[j * per_m:(j + 1) * per_m])
            res["per_m"][f"m{m}"] = {"us": round(us, 3), "weight_gbs": round(wb / us / 1e3, 1)}
        return label, res

    out = dict([
        one("no_prefetch"),
        one("in_launch_next_weight_15pct_l2", frac=0.15),
        one("side_stream_50pct_l2_joined", side_frac=0.5, join=True),
        one("side_stream_15pct_l2_joined", side_frac=0.15, join=True),
        one("side_stream_50pct_l2_unjoined", side_frac=0.5, join=False),
    ])
    set_next(0.0)
    wl.bind_streams([torch_stream])
    out["captured_graph"] = chain_graph(wl, torch_stream, steps)
    out["captured_graph_side_stream_50pct_l2"] = chain_graph(wl, torch_stream, steps, side_frac=0.5)
    out["group_launch_per_m_ordered"] = chain_groups(wl, s, torch_stream, steps)
    out["router_and_latent_as_one_launch"] = chain_router_latent(wl, s, torch_stream, steps)
    return out


def chain_router_latent(wl, s, torch_stream, steps):
    """The chain with its router-score GEMM and latent input projection,
    which read the same hidden state, as one group launch without ordering
    (the single-GPU form of the pages' router + latent projection as one
    GEMM); the other three projections as their own launches.  Both read the
    router stage's x here."""
    import torch
    from projection_gemm_gb300 import inputs as I
    from projection_gemm_gb300 import skg
    per_m = len(I.CHAIN_STAGES)
    pairs = []
    try:
        for j, m in enumerate(I.CHAIN_M):
            r, l = wl.ops[j * per_m + 2], wl.ops[j * per_m + 3]
            g = skg.Group(m, [r["p"].N, l["p"].N], [r["p"].K, l["p"].K], [r["p"].epilogue, l["p"].epilogue], None)
            pairs.append((g, [r["args"][0]] * 2, [r["args"][1], l["args"][1]], [r["args"][3], l["args"][3]]))

        def step(events=None):
            for j in range(len(I.CHAIN_M)):
                if events is not None:
                    events[j].record(torch_stream)
                base = j * per_m
                for i in (0, 1):
                    wl.launch(wl.ops[base + i], s)
                g, xs, ws, ys = pairs[j]
                skg.skg_group_run(g.handle, xs, ws, None, ys, s)
                wl.launch(wl.ops[base + 4], s)
            if events is not None:
                events[-1].record(torch_stream)
        for _ in range(3):
            step()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(torch_stream)
        for _ in range(steps):
            step()
        b.record(torch_stream)
        torch.cuda.synchronize()
        el = a.elapsed_time(b) / 1e3
        seg_us = [[] for _ in I.CHAIN_M]
        for _ in range(12):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(I.CHAIN_M) + 1)]
            step(ev)
            torch.cuda.synchronize()
            for j in range(len(I.CHAIN_M)):
                seg_us[j].append(ev[j].elapsed_time(ev[j + 1]) * 1e3)
        res = {"us_per_step": round(el / steps * 1e6, 3), "gbs": round(wl.weight_bytes() * steps / el / 1e9, 1),
               "per_m": {}}
        for j, m in enumerate(I.CHAIN_M):
            us = statistics.median(seg_us[j])
            wb = sum(o["p"].weight_bytes() for o in wl.ops[j * per_m:(j + 1) * per_m])
            res["per_m"][f"m{m}"] = {"us": round(us, 3), "weight_gbs": round(wb / us / 1e3, 1)}
        for g, *_ in pairs:
            g.check()
        return res
    finally:
        for g, *_ in pairs:
            g.close()


def chain_groups(wl, s, torch_stream, steps):
    """The chain with each M's five projections as one group launch
    (skg_group), each projection ordered after the previous one."""
    import torch
    from projection_gemm_gb300 import inputs as I
    from projection_gemm_gb300 import skg
    per_m = len(I.CHAIN_STAGES)
    groups = []
    try:
        for j, m in enumerate(I.CHAIN_M):
            seg = wl.ops[j * per_m:(j + 1) * per_m]
            g = skg.Group(m, [o["p"].N for o in seg], [o["p"].K for o in seg], [o["p"].epilogue for o in seg],
                          [0] + [1] * (per_m - 1))
            groups.append((g, [[o["args"][i] for o in seg] for i in range(4)]))

        def step(events=None):
            for j, (g, (xs, ws, rs, ys)) in enumerate(groups):
                if events is not None:
                    events[j].record(torch_stream)
                skg.skg_group_run(g.handle, xs, ws, rs, ys, s)
            if events is not None:
                events[-1].record(torch_stream)
        for _ in range(3):
            step()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(torch_stream)
        for _ in range(steps):
            step()
        b.record(torch_stream)
        torch.cuda.synchronize()
        el = a.elapsed_time(b) / 1e3
        seg_us = [[] for _ in groups]
        for _ in range(12):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(groups) + 1)]
            step(ev)
            torch.cuda.synchronize()
            for j in range(len(groups)):
                seg_us[j].append(ev[j].elapsed_time(ev[j + 1]) * 1e3)
        res = {"us_per_step": round(el / steps * 1e6, 3), "gbs": round(wl.weight_bytes() * steps / el / 1e9, 1),
               "per_m": {}}
        for j, m in enumerate(I.CHAIN_M):
            us = statistics.median(seg_us[j])
            wb = sum(o["p"].weight_bytes() for o in wl.ops[j * per_m:(j + 1) * per_m])
            res["per_m"][f"m{m}"] = {"us": round(us, 3), "weight_gbs": round(wb / us / 1e3, 1),
                                     "grid": groups[j][0].info()["grid"]}
        for g, _ in groups:
            g.check()
        return res
    finally:
        for g, _ in groups:
            g.close()


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    from projection_gemm_gb300 import build as B
    from projection_gemm_gb300 import skg

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    B.build()
    skg.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    peak_hbm, peak_tf, peak_src = load_peaks()
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    wl = DeviceWorkload(args.workload, dev, pdl=bool(args.pdl), keep_host=True, host_bits=want_cpu)
    wl.bind_streams([stream])
    launches_per_step = len(wl.ops)
    wbytes_step = wl.weight_bytes()

    warm = max(3, args.warmup)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(warm):
        wl.step(s)
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / warm
    K = args.steps if args.steps else max(20, min(40000, int(args.seconds / max(est, 1e-6))))

    clocks = ClockSampler(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.5)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    # ---- timed region: exactly K steps, events only at its two ends
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    start.record(stream)
    for _ in range(K):
        wl.step(s)
    end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    if world > 1:
        dist.barrier()
    elapsed = start.elapsed_time(end) / 1e3
    max_t, total_bytes = aggregate(elapsed, wbytes_step * K, world)
    value = total_bytes / max_t / 1e9

    # ---- separate passes after the timed region
    p0 = time.time()
    b2b = measure_back_to_back(wl, s, stream, l2_bytes)
    iso = measure_event_isolated(wl, s, stream)
    table = projection_table(wl, b2b, iso, peak_hbm, peak_tf)
    kinds = measure_kind_runs(wl, s, stream)
    for k in kinds.values():
        k["frac"] = round(k["gbs"] / peak_hbm, 4)
    p1 = time.time()

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": warm, "ms_per_step": round(max_t / K * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.desc, **wl.cfg, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": ("inputs larger than L2: every step streams %.1f MB of distinct weights" % (wbytes_step / 1e6)),
                   "pdl": bool(args.pdl), "launch": "eager skg_run calls",
                   "timed_region": "exactly `steps` steps, CUDA events only at its two ends"},
        "per_projection": table,
        "roofline": roofline_from(table, wl, peak_hbm, peak_src, args.workload),
        "kernel_in_step": kinds,
        "gpu_launches": launches_per_step * K,
    }
    bars = [r for r in table.values() if "bar" in r]
    result["projections_meeting_bar"] = f"{sum(r['meets_bar'] for r in bars)}/{len(bars)}"

    # ---- e2e: activations from pinned host memory, outputs back, every step
    if not args.no_e2e:
        graph = full = None
        if args.e2e_launch == "graph":
            cap = torch.cuda.Stream(device=dev)
            cap.wait_stream(stream)
            wl.bind_streams([stream, cap])
            with torch.cuda.stream(cap):
                wl.step(cap.cuda_stream)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                wl.step(cap.cuda_stream)
            torch.cuda.synchronize()
            # the whole step, copies included: one graph launch per step
            cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
            with torch.cuda.stream(cap):
                wl.e2e_step(cap, cin, cout)
            torch.cuda.synchronize()
            full = torch.cuda.CUDAGraph()
            with torch.cuda.graph(full, stream=cap):
                wl.e2e_step(cap, cin, cout)
            torch.cuda.synchronize()
            wl.bind_streams([stream])
        Ke = max(3, min(K, int(args.e2e_seconds / max(est, 1e-6))))
        h2d, d2h = wl.host_in.numel(), wl.host_out.numel()

        def e2e_step():
            if full is not None:
                full.replay()
            else:
                wl.dev_in.copy_(wl.host_in, non_blocking=True)
                wl.step(s)
                wl.host_out.copy_(wl.dev_out, non_blocking=True)
            stream.synchronize()
        for _ in range(3):
            e2e_step()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(Ke):
            e2e_step()
        te = time.perf_counter() - t0
        if not torch.equal(wl.host_out, wl.dev_out.cpu()):
            raise RuntimeError("end-to-end step: the outputs copied back differ from the device's")
        te, eb = aggregate(te, wbytes_step * Ke, world)
        result["e2e"] = {"value": round(eb / te / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                         "d2h_bytes_per_step": d2h, "steps": Ke,
                         "ms_per_step": round(te / Ke * 1e3, 4),
                         "launch": ("each step's input copies, skg_run calls and output copies captured once "
                                    "as one CUDA graph, replayed every step: the first projection's inputs "
                                    "copied first, the rest beside its kernel; each output copied back as "
                                    "soon as its projection completes" if full is not None else
                                    "eager skg_run calls between the copies"),
                         "sync": "host waits for every step's output copy before the next step"}
        if graph is not None and world == 1:
            result["e2e"]["pipelined"] = e2e_pipelined(wl, stream, Ke, wbytes_step)
        del graph, full

    host = wl.host
    wl.close()
    del wl
    torch.cuda.empty_cache()

    # ---- the other named workloads
    c0 = time.time()
    if not args.headline_only and rank == 0:
        result["configs"] = {}
        for name in EXTRA_CONFIGS:
            if name == args.workload:
                continue
            result["configs"][name] = measure_config(name, dev, s, stream, args, peak_hbm, peak_tf, l2_bytes)
            torch.cuda.empty_cache()
    c1 = time.time()
    if clocks:
        time.sleep(0.2)
        clocks.stop()
        result["clocks"] = clocks.summary([(w0, w1), (p0, p1), (c0, c1)])
        result["clocks"]["window"] = "timed region and the measurement passes after it"
        result["clocks"]["samples_in_timed_region"] = clocks.summary([(w0, w1)])["samples"]

    if want_cpu:
        smp = OracleSample(host, args.cpu_seconds)
        gbs, secs = smp.run()
        result["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": smp.cores, "kind": "oracle",
                                  "sample": smp.desc, "seconds": round(secs, 2)}
    if world > 1:
        dist.destroy_process_group()
    return result if rank == 0 else None


# ------------------------------------------------------------ reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    projs, desc, cfg = workload(args.workload)
    K = args.steps or 5
    warm = max(3, args.warmup)
    smp = OracleSample(host_data(projs), min(20.0, max(0.5, args.ref_seconds / K)))
    for _ in range(warm):
        smp.run_rows(16)
    vals, secs, wbytes = [], 0.0, 0.0
    for _ in range(K):
        g, dt = smp.run()
        vals.append(g)
        secs += dt
        wbytes += g * dt * 1e9
    value = wbytes / secs / 1e9 if secs > 0 else statistics.median(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": warm, "ms_per_step": round(secs / K * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, **cfg, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": smp.cores, "kind": "oracle",
                         "sample": smp.desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (default: about --seconds of work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=("sweep", "chain", "wide", "deepk", "pr1"), default="sweep")
    ap.add_argument("--seconds", type=float, default=3.0, help="target timed-region length")
    ap.add_argument("--e2e-seconds", type=float, default=1.5)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--pdl", type=int, default=1)
    ap.add_argument("--e2e-launch", choices=("graph", "eager"), default="graph",
                    help="how the end-to-end leg issues a step's launches between its host copies")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other named workloads (wide, deep-K, PR1, chain)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    args = ap.parse_args(argv)
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        line = json.dumps(res)
        print(line, flush=True)
        if args.out:
            with open(args.out, "a") as f:
                f.write(line + "\n")


if __name__ == "__main__":
    main()
