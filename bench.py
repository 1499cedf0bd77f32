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
  chain            the five projections of a decode layer at M = 1, 8, 64,
                   each launch asking the L2 for the start of the next weight.
  wide / deepk     the wide input projection and the deep-K output projection
                   with residual, at their M values.

`value` is the whole job's weight bytes / device time (CUDA events around the
timed steps, max over ranks).  `e2e` repeats the measurement through the
public API with the step's activations copied from pinned host memory and its
outputs copied back inside the timed region (weights stay resident: they are
parameters, not per-step inputs).  `--impl reference` times the CPU oracle on
the same metric instead (a bounded sample of each step).
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
                       "7168->384 (fp32), 7168->4096, 4096->7168 (+res); each launch asks the L2 "
                       "for the start of the next W"), {"M": list(I.CHAIN_M), "stages": [list(s) for s in I.CHAIN_STAGES]}
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
    """nvidia-smi samples (200 ms) while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = [s for t, s in self.samples if self.t0 is not None and self.t0 - 0.1 <= t <= self.t1 + 0.25]
        if not rows and self.samples:
            rows = [self.samples[-1][1]]
        sm, mx, reasons, power = [], None, set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
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
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


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


class GroupProjection:
    """Several projections launched as one group: the bench's per-launch
    figures (weight and algorithmic bytes, flops) summed over its members."""

    def __init__(self, members):
        self.members = members
        self.M = members[0].M
        self.N = [p.N for p in members]
        self.K = [p.K for p in members]
        self.name = f"{members[0].name}..{members[-1].name}"

    def weight_bytes(self):
        return sum(p.weight_bytes() for p in self.members)

    def algorithmic_bytes(self):
        return sum(p.algorithmic_bytes() for p in self.members)

    def flops(self):
        return sum(p.flops() for p in self.members)


def make_group(members, ordered=True):
    from projection_gemm_gb300 import skg
    ps = [o["p"] for o in members]
    g = skg.Group(ps[0].M, [p.N for p in ps], [p.K for p in ps], [p.epilogue for p in ps],
                  [0] + [1 if ordered else 0] * (len(ps) - 1))
    info = g.info()
    return dict(p=GroupProjection(ps), group=g, plans=[o["plan"] for o in members],
                info={"kernel": "splitk_group", "split_k": info["split"], "prefetch_bytes": 0,
                      "grid": info["grid"], "stages": info["stages"]},
                x=[o["x"] for o in members], W=[o["W"] for o in members], res=[o["res"] for o in members],
                y=[o["y"] for o in members])


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    from projection_gemm_gb300 import build as B
    from projection_gemm_gb300 import skg
    from projection_gemm_gb300.inputs import generate

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
    projs, desc, cfg = workload(args.workload)
    peak_hbm, peak_tf, peak_src = load_peaks()

    # Operands resident in HBM.  A step's activations (x, residual) and its
    # outputs each live in one packed buffer (256-byte aligned segments), so
    # the end-to-end run moves them with one host->device and one
    # device->host copy per step.
    def seg(nbytes):
        return (nbytes + 255) // 256 * 256
    gens = [generate(p) for p in projs]
    in_bytes = sum(seg(t.x.numel() * 2) + (seg(t.res.numel() * 2) if t.res is not None else 0) for t in gens)
    out_bytes = sum(seg(p.M * p.N * p.out_bytes_per_elem) for p in projs)
    dev_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    dev_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    host_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()

    def view(buf, off, shape, dt):
        n = shape[0] * shape[1] * torch.empty((), dtype=dt).element_size()
        return buf[off:off + n].view(dt).view(*shape)

    ops, hostcopy = [], []
    oi = oo = 0
    for p, t in zip(projs, gens):
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            from projection_gemm_gb300.inputs import bits
            hostcopy.append((p, bits(t.x), bits(t.W), None if t.res is None else bits(t.res)))
        plan = skg.Plan(p.M, p.N, p.K, p.epilogue)
        plan.set_pdl(bool(args.pdl))
        dt = torch.float32 if p.epilogue == "fp32" else torch.bfloat16
        x = view(dev_in, oi, (p.M, p.K), torch.bfloat16)
        view(host_in, oi, (p.M, p.K), torch.bfloat16).copy_(t.x)
        oi += seg(t.x.numel() * 2)
        res = None
        if t.res is not None:
            res = view(dev_in, oi, (p.M, p.N), torch.bfloat16)
            view(host_in, oi, (p.M, p.N), torch.bfloat16).copy_(t.res)
            oi += seg(t.res.numel() * 2)
        y = view(dev_out, oo, (p.M, p.N), dt)
        oo += seg(p.M * p.N * p.out_bytes_per_elem)
        ops.append(dict(p=p, plan=plan, info=plan.info(), x=x, W=t.W.to(dev), res=res, y=y))
    dev_in.copy_(host_in)
    del gens
    # [PF] on a side stream (--prefetch f): a prefetch kernel fills the L2
    # with the next projection's weight while the current one runs.
    side_pf = args.prefetch is not None and args.prefetch > 0
    side = torch.cuda.Stream(device=dev)
    stream = torch.cuda.current_stream(dev)
    if args.prefetch is not None:
        for o in ops:
            skg.skg_plan_set_prefetch_fraction(o["plan"].handle, max(0.0, args.prefetch))

    # [PF] inside the launch: each projection also asks the L2 for the first
    # part of the weight that runs after it (the step wraps around).
    next_frac = args.next_weight if args.next_weight is not None else (0.15 if args.workload == "chain" else 0.0)
    if next_frac > 0:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        for i, o in enumerate(ops):
            nxt = ops[(i + 1) % len(ops)]
            o["plan"].set_next_weight(nxt["W"], int(min(nxt["p"].weight_bytes(), next_frac * l2)))

    # --fused: each run of consecutive projections with the same M >= --fused-min-m is
    # one group launch (skg_group), every projection after the first ordered
    # after the previous one (dep), as consecutive launches are -- or, with
    # --fused-order independent, with no order among them.
    if args.fused:
        side_pf = False
        segs, i = [], 0
        while i < len(ops):
            j = i + 1
            while ops[i]["p"].M >= args.fused_min_m and j < len(ops) and ops[j]["p"].M == ops[i]["p"].M:
                j += 1
            single = j == i + 1 and not (args.fused_single and ops[i]["p"].M >= args.fused_min_m)
            segs.append(ops[i] if single else make_group(ops[i:j], args.fused_order == "chain"))
            i = j
        ops = segs

    # Runs of consecutive launches of one kernel kind: events at their
    # boundaries time each kind's launches without splitting the runs.
    groups, g0 = [], 0
    for i in range(1, len(ops) + 1):
        if i == len(ops) or ops[i]["info"]["kernel"] != ops[g0]["info"]["kernel"]:
            groups.append((g0, i))
            g0 = i
    group_start = {a: j for j, (a, _) in enumerate(groups)}

    def launch(o, s):
        if "group" in o:
            o["group"].run(o["x"], o["W"], o["res"], o["y"], s)
        else:
            o["plan"].run(o["x"], o["W"], o["res"], o["y"], s)

    def step(events=None, mode="launch", s=None):
        s = stream if s is None else s
        for i, o in enumerate(ops):
            if side_pf and i + 1 < len(ops) and ops[i + 1]["info"]["prefetch_bytes"] > 0:
                side.wait_stream(s)
                ops[i + 1]["plan"].prefetch(ops[i + 1]["W"], side)
            if events is not None and (mode == "launch" or i in group_start):
                events[i if mode == "launch" else group_start[i]].record(s)
            launch(o, s)
            if side_pf and i + 1 < len(ops):
                s.wait_stream(side)
        if events is not None:
            events[-1].record(s)

    launches_per_step = len(ops) + (sum(1 for o in ops[1:] if o["info"]["prefetch_bytes"] > 0) if side_pf else 0)
    wbytes_step = sum(o["p"].weight_bytes() for o in ops)

    warm = max(3, args.warmup)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(warm):
        step()
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / warm
    # --graph: a step's launches captured once into a CUDA graph (skg_run
    # allocates nothing; the programmatic launch edges are kept, and a
    # side-stream prefetch becomes a forked node joined before the next
    # projection) and replayed each step, so the host issues one launch per
    # step.  Steps that carry events run eagerly.
    graph = None
    if args.graph or (args.e2e_launch == "graph" and not args.no_e2e):
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            step(s=cap)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            step(s=cap)   # the side stream forks from and joins back into the capture
        side.wait_stream(stream)
        torch.cuda.synchronize()
        for _ in range(warm):
            graph.replay()
        torch.cuda.synchronize()
    K = args.steps if args.steps else max(20, min(40000, int(args.seconds / max(est, 1e-6))))
    # Sampled steps carry events, alternately before every launch (the
    # us/projection figures) or at kernel-kind boundaries only (each kind's
    # launch durations, with the programmatic overlap inside a run intact).
    # An event between two launches ends their overlap, so only about 300 of
    # the K steps carry any.
    sample_every = max(1, K // 300)
    sampled = list(range(0, K, sample_every))
    modes = {k: ("launch" if j % 2 == 0 else "group") for j, k in enumerate(sampled)}
    evs = {k: [torch.cuda.Event(enable_timing=True)
               for _ in range((len(ops) if modes[k] == "launch" else len(groups)) + 1)] for k in sampled}

    clocks = ClockSampler(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.6)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    start.record(stream)
    for k in range(K):
        if args.graph and k not in evs:
            graph.replay()
        else:
            step(evs.get(k), modes.get(k, "launch"))
    end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    if world > 1:
        dist.barrier()
    if clocks:
        time.sleep(0.3)
        clocks.stop()
        clocks.window(w0, w1)
    elapsed = start.elapsed_time(end) / 1e3
    max_t, total_bytes = aggregate(elapsed, wbytes_step * K, world)
    value = total_bytes / max_t / 1e9

    # per-launch durations from the sampled steps (events on the launch stream)
    per = {i: [] for i in range(len(ops))}
    kern = {}
    for k in sampled:
        e = evs[k]
        if modes[k] == "launch":
            for i in range(len(ops)):
                per[i].append(e[i].elapsed_time(e[i + 1]) * 1e3)  # us
            continue
        for j, (a, b) in enumerate(groups):
            kk = kern.setdefault(ops[a]["info"]["kernel"], {"bytes": 0.0, "us": 0.0, "launches": 0})
            kk["bytes"] += sum(ops[i]["p"].algorithmic_bytes() for i in range(a, b))
            kk["us"] += e[j].elapsed_time(e[j + 1]) * 1e3
            kk["launches"] += b - a
    per_m = {}
    for i, o in enumerate(ops):
        p = o["p"]
        us = statistics.median(per[i])
        t_ideal = max(p.algorithmic_bytes() / (peak_hbm * 1e9), p.flops() / (peak_tf * 1e12)) * 1e6
        key = f"{p.name}"
        per_m[key] = {"M": p.M, "N": p.N, "K": p.K, "kernel": o["info"]["kernel"], "split": o["info"]["split_k"],
                      "us": round(us, 3), "weight_gbs": round(p.weight_bytes() / us / 1e3, 1),
                      "roofline_frac": round(t_ideal / us, 4)}
        if "grid" in o["info"]:
            per_m[key].update(grid=o["info"]["grid"], stages=o["info"]["stages"])
    dom = max(kern, key=lambda k: kern[k]["us"])
    achieved = kern[dom]["bytes"] / (kern[dom]["us"] * 1e-6) / 1e9
    traffic = kernel_traffic(dom, args.workload)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak_hbm, "unit": "GB/s",
                "frac": round(achieved / peak_hbm, 4), "traffic": traffic,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback",
                "launches_timed": kern[dom]["launches"],
                "timing": "events at the boundaries of each run of this kernel's launches in sampled steps"}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": warm, "ms_per_step": round(max_t / K * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": desc, **cfg, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": ("inputs larger than L2: every step streams %.1f MB of distinct weights" % (wbytes_step / 1e6)),
                   "pdl": bool(args.pdl),
                   "fused_groups": bool(args.fused),
                   **({"fused_order": ("each projection of a group after the previous one" if args.fused_order == "chain"
                                       else "the projections of a group independent of one another"),
                       "fused_min_m": args.fused_min_m}
                      if args.fused else {}),
                   "launch": ("cuda graph of the step's launches, replayed (steps carrying events run eagerly)"
                              if args.graph else "eager skg_run calls"),
                   "next_weight_l2_fraction": next_frac,
                   "side_stream_prefetch_fraction": args.prefetch if side_pf else 0.0},
        "per_projection": per_m, "roofline": roofline,
        "gpu_launches": launches_per_step * K,
    }
    if clocks:
        result["clocks"] = clocks.summary()

    # e2e: activations from pinned host memory, outputs back, every step
    if not args.no_e2e:
        Ke = max(3, min(K, int(args.e2e_seconds / max(est, 1e-6))))
        h2d, d2h = host_in.numel(), host_out.numel()

        def e2e_step():
            dev_in.copy_(host_in, non_blocking=True)
            if args.e2e_launch == "graph":
                graph.replay()
            else:
                step()
            host_out.copy_(dev_out, non_blocking=True)
            stream.synchronize()
        for _ in range(2):
            e2e_step()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(Ke):
            e2e_step()
        te = time.perf_counter() - t0
        te, eb = aggregate(te, wbytes_step * Ke, world)
        result["e2e"] = {"value": round(eb / te / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                         "d2h_bytes_per_step": d2h, "steps": Ke,
                         "ms_per_step": round(te / Ke * 1e3, 4),
                         "launch": ("each step's skg_run calls captured once as a CUDA graph and replayed "
                                    "between the copies" if args.e2e_launch == "graph" else
                                    "eager skg_run calls between the copies"),
                         "sync": "host waits for every step's output copy before the next step"}

    for o in ops:
        (o["group"] if "group" in o else o["plan"]).check()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSample(hostcopy, args.cpu_seconds)
        gbs, secs = smp.run()
        result["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": smp.cores, "kind": "oracle",
                                  "sample": smp.desc, "seconds": round(secs, 2)}
    for o in ops:
        if "group" in o:
            o["group"].close()
            for pl in o["plans"]:
                pl.close()
        else:
            o["plan"].close()
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
    ap.add_argument("--graph", type=int, default=0,
                    help="1: replay each step as one captured CUDA graph (measured slower: replays do not overlap)")
    ap.add_argument("--e2e-launch", choices=("graph", "eager"), default="graph",
                    help="how the end-to-end leg issues a step's launches between its host copies")
    ap.add_argument("--prefetch", type=float, default=None,
                    help="fraction of L2 filled with the next weight by a kernel on a side stream (default: off)")
    ap.add_argument("--next-weight", type=float, default=None,
                    help="fraction of L2 of the next projection's weight each launch asks the L2 for "
                         "(default: 0.15 for the chain, off otherwise)")
    ap.add_argument("--fused", type=int, default=0,
                    help="1: consecutive projections of one M (>= --fused-min-m) as one group launch (skg_group)")
    ap.add_argument("--fused-order", choices=("chain", "independent"), default="chain",
                    help="with --fused: order each projection after the previous one (as consecutive launches "
                         "are), or run a group's projections as independent work (e.g. projections of one x)")
    ap.add_argument("--fused-min-m", type=int, default=3,
                    help="with --fused: the smallest M whose projections are grouped (M <= 2 groups run the "
                         "split-K kernel, in place of the GEMV)")
    ap.add_argument("--fused-single", type=int, default=0,
                    help="with --fused: a projection with no same-M neighbour also runs as a "
                         "one-projection group (units handed out dynamically)")
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
