"""Fill the picker table from timings taken on the GPU.

For every projection shape of the workloads (the batch sweep, the wide and
deep-K projections and the five decode-layer chain stages) and every M they
are run at, each candidate launch configuration inside the kernel kind that
M selects is timed back to back -- the way a decode step issues projections
-- over enough distinct copies of the weight that no launch finds its weight
in L2.  The fastest candidate becomes a row of csrc/skg_plan_table.inc; the
full log is written as JSON beside it.

usage: python -m projection_gemm_gb300.tune [--out-inc PATH] [--out-log PATH] [--rounds R]
Rebuild the library afterwards (the table is compiled in).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import time

import torch

from . import build, skg
from .inputs import CHAIN_M, CHAIN_STAGES, DEEPK_M, SWEEP_M, WIDE_M, Projection, generate

HERE = os.path.dirname(os.path.abspath(__file__))
NOMINAL_HBM_BPS = 8.0e12   # no launch can stream its weight faster than the HBM
INC = os.path.join(HERE, "csrc", "skg_plan_table.inc")
REDUCER_SHAPES = 6         # fastest launch shapes of a split-K row also timed at each reducer count


def shapes():
    """(N, K, epilogue) -> the M values it runs at."""
    out = {}
    def add(N, K, epi, ms):
        out.setdefault((N, K, epi), set()).update(ms)
    add(7168, 7168, "bf16", SWEEP_M)
    add(12288, 7168, "bf16", WIDE_M)
    add(7168, 16384, "bf16_residual", DEEPK_M)
    for K, N, epi in CHAIN_STAGES:
        add(N, K, epi, CHAIN_M)
    return {k: sorted(v) for k, v in out.items()}


def candidates(M, N, K):
    """Every candidate names its kernel kind: a plan's default kind follows the
    table being replaced, so a candidate must not depend on it."""
    if M <= 2:
        c = [{"split_k": 1, "stages": 1, "ahead": a} for a in (0, 1, 2)]
        c += [{"split_k": 1, "stages": 2, "tma_burst": b, "ahead": 0} for b in (4, 8)]
        c += [{"split_k": 1, "stages": 3, "tma_burst": b, "ahead": a} for b in (4, 8) for a in (0, 1, 2)]
        for split in (2, 4, 8):
            for ring in (2, 3, 4):
                c.append({"split_k": split, "stages": ring, "ahead": 0})
        for cfg in c:
            cfg["kind"] = skg.SKG_KERNEL_GEMV
        # the tensor-core kernel with the tokens padded to 16 columns
        c += [{"kind": skg.SKG_KERNEL_SPLITK_TC, "split_k": sp, "stages": st, "ahead": a}
              for sp in (2, 4, 8) for st in (4, 5, 6) for a in (0, 2)]
        return c
    # ahead up to a CTA's whole K range: the next launch's weight requests
    # can cover the previous launch's tail
    return [{"split_k": s, "stages": st, "ahead": a} for s in (2, 4, 8, 16) for st in (3, 4, 5, 6)
            for a in (0, 2, 4, 8, 12, 16, 24, 32)]


def read_rows(path):
    """The rows of an existing table file, as the tuple main() writes:
    (kind, M, N, K, epilogue, split, stages, grid, aux, ahead, reducers, us,
    GB/s); a row without the reducers column reads as 0 (library default)."""
    rows = []
    pat = re.compile(r"^\{([-\d, ]+)\},\s*// ([\d.]+) us, ([\d.]+) GB/s")
    for line in open(path):
        m = pat.match(line)
        if m:
            ints = tuple(int(v) for v in m.group(1).split(","))
            if len(ints) == 10:
                ints += (0,)
            rows.append(ints + (float(m.group(2)), float(m.group(3))))
    return rows


def time_config(M, N, K, epi, cfg, Ws, x, res, y, rounds):
    """Launch time per projection: one round over every weight copy is
    captured in a CUDA graph and replayed `rounds` times (no host launch
    cost in the measurement; programmatic dependent launch stays on)."""
    p = None
    try:
        p = skg.Plan(M, N, K, epi)
        if cfg.get("kind"):
            p.force_kernel(cfg["kind"])
        force = {k: v for k, v in cfg.items() if k in ("split_k", "stages", "tma_burst") and v}
        p.force(**force)
        p.set_l2_ahead(cfg.get("ahead", 0))
        if cfg.get("reducers"):
            p.set_reducers(cfg["reducers"])
        for W in Ws[:2]:
            p.run(x, W, res, y)             # descriptors, attributes: outside the capture
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for W in Ws:
                p.run(x, W, res, y, s)
        # replay() launches on the current stream: time on that stream
        g.replay()
        torch.cuda.synchronize()
        main = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        for _ in range(rounds):
            g.replay()
        b.record(main)
        torch.cuda.synchronize()
        p.check()
        us = a.elapsed_time(b) * 1e3 / (rounds * len(Ws))
        if 2 * N * K / (us * 1e-6) > NOMINAL_HBM_BPS:
            raise RuntimeError(f"implausible timing {us:.3f} us for {2 * N * K} weight bytes")
        return us, p.info()
    except skg.SkgError:
        return None, None
    finally:
        if p is not None:
            p.close()


def row_config(row):
    """A table row as the candidate dict time_config takes."""
    kind, M, N, K, epi, split, stages, grid, aux, ahead, reducers = row[:11]
    cfg = {"kind": kind, "split_k": split, "stages": stages, "ahead": ahead}
    if kind == skg.SKG_KERNEL_SPLITK_TC:
        if aux > 1:
            cfg["tma_burst"] = aux
        if reducers:
            cfg["reducers"] = reducers
    elif split == 1 and stages >= 2:
        cfg["tma_burst"] = aux
    return cfg


def measured_hbm_gbs():
    """The measured copy bandwidth of this GPU, else the nominal 8 TB/s."""
    try:
        with open(os.path.join(os.path.dirname(HERE), "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"])
    except Exception:
        return NOMINAL_HBM_BPS / 1e9


# Projections that always run as one fixed sequence: each workload's step.
SEQUENCES = {
    "sweep": lambda: [(M, 7168, 7168, "bf16") for M in SWEEP_M],
    "chain": lambda: [(M, N, K, epi) for M in CHAIN_M for (K, N, epi) in CHAIN_STAGES],
    "wide": lambda: [(M, 12288, 7168, "bf16") for M in WIDE_M],
    "deepk": lambda: [(M, 7168, 16384, "bf16_residual") for M in DEEPK_M],
}


def sequence_refine(rows, log, names=("sweep",), steps=150, reps=3, margin_us=0.4, keep=8, bar_margin=0.02,
                    passes=2):
    """The projections of a workload's step always run as one sequence (the
    batch sweep M = 1, 2, ..., 64; the decode layer's five stages at M = 1, 8,
    64; the wide and deep-K batches), and a launch's best configuration alone
    is not always its best next to the others: a neighbour with another
    shared-memory footprint starts later, and the next launch's look-ahead
    requests meet this launch's latency-bound reduction in L2.  Coordinate
    descent over each projection's `keep` fastest launch shapes alone (with
    look-ahead 0 to 4 each), timing whole eager steps of every named
    workload that holds the projection (a shape shared by two workloads, such
    as the 12288-wide projection of the chain and of the wide batch, is
    judged by the sum of their steps); a change is kept only if it beats the
    incumbent, timed alternately, by margin_us in every one of `reps` pairs,
    and only among launch shapes whose time alone still clears the
    projection's roofline bar (0.80 at M <= 16, 0.70 above) by bar_margin.
    Returns the rows with the sequences' entries replaced."""
    if isinstance(names, str):
        names = (names,)
    byKey = {(r[1], r[2], r[3], r[4]): r for r in rows}
    seq_keys = {n: [(M, N, K, skg.EPILOGUES[epi]) for M, N, K, epi in SEQUENCES[n]()] for n in names}
    keys = []
    for n in names:
        keys += [k for k in seq_keys[n] if k not in keys]
    holders = {k: [n for n in names if k in seq_keys[n]] for k in keys}
    epi_name = {v: k for k, v in skg.EPILOGUES.items()}
    cands = {}
    for key in keys:
        M, N, K, e = key
        entries = sorted((x for x in log if (x["M"], x["N"], x["K"], skg.EPILOGUES[x["epilogue"]]) == key
                          and (M > 2 or "kind" in x["config"])), key=lambda x: x["us"])
        shapes_, c, seen = [], [], set()
        for x in entries:
            shape = json.dumps({k: v for k, v in x["config"].items() if k != "ahead"}, sort_keys=True)
            if shape not in shapes_:
                shapes_.append(shape)
        for shape in shapes_[:keep]:
            for x in entries:
                cfg = x["config"]
                ck = json.dumps(cfg, sort_keys=True)
                if (json.dumps({k: v for k, v in cfg.items() if k != "ahead"}, sort_keys=True) == shape
                        and cfg.get("ahead", 0) <= 4 and ck not in seen):
                    seen.add(ck)
                    c.append((cfg, x["us"]))
        bar = (0.80 if M <= 16 else 0.70) + bar_margin
        ideal_us = Projection(M, N, K, epi_name[e]).algorithmic_bytes() / (measured_hbm_gbs() * 1e3)
        cands[key] = [(cfg, us) for cfg, us in c if ideal_us / us >= bar]
    ops = {}
    for n in names:
        ops[n] = []
        for i, (M, N, K, epi) in enumerate(SEQUENCES[n]()):
            t = generate(Projection(M, N, K, epi, seed=950 + i))
            ops[n].append(dict(W=t.W.cuda(), x=t.x.cuda(), res=None if t.res is None else t.res.cuda(),
                               y=torch.empty(M, N, dtype=torch.float32 if epi == "fp32" else torch.bfloat16,
                                             device="cuda")))

    def plan_for(key, cfg):
        M, N, K, e = key
        p = skg.Plan(M, N, K, epi_name[e])
        if cfg.get("kind"):
            p.force_kernel(cfg["kind"])
        force = {k: v for k, v in cfg.items() if k in ("split_k", "stages", "tma_burst") and v}
        p.force(**force)
        p.set_l2_ahead(cfg.get("ahead", 0))
        if cfg.get("reducers"):
            p.set_reducers(cfg["reducers"])
        return p

    def step_us(plans, n):
        def one():
            for key, o in zip(seq_keys[n], ops[n]):
                plans[key].run(o["x"], o["W"], o["res"], o["y"])
        for _ in range(3):
            one()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            one()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / steps

    def total_us(plans, ns):
        return sum(step_us(plans, n) for n in ns)

    choice = {k: row_config(byKey[k]) for k in keys}
    us_alone = {k: byKey[k][11] for k in keys}
    plans = {k: plan_for(k, choice[k]) for k in keys}
    for n in names:
        print(f"{n} step with the table: {step_us(plans, n):.2f} us", flush=True)
    for _ in range(passes):
        for key in keys:
            ns = holders[key]
            for cfg, us in cands[key]:
                if cfg == choice[key]:
                    continue
                try:
                    trial = plan_for(key, cfg)
                except skg.SkgError:
                    continue
                incumbent = plans[key]
                wins = 0
                for _ in range(reps):
                    plans[key] = incumbent
                    t_inc = total_us(plans, ns)
                    plans[key] = trial
                    t_new = total_us(plans, ns)
                    wins += t_new < t_inc - margin_us
                if wins == reps:
                    incumbent.close()
                    choice[key], us_alone[key] = cfg, us
                    print(f"  {key}: {cfg} ({t_new:.2f} against {t_inc:.2f} us, steps {'+'.join(ns)})", flush=True)
                else:
                    trial.close()
                    plans[key] = incumbent
    for n in names:
        print(f"{n} step chosen in sequence: {step_us(plans, n):.2f} us", flush=True)
    for p in plans.values():
        p.close()
    out = []
    for r in rows:
        key = (r[1], r[2], r[3], r[4])
        if key in choice:
            cfg = choice[key]
            M, N, K = key[:3]
            kind = cfg.get("kind", skg.SKG_KERNEL_GEMV if M <= 2 else skg.SKG_KERNEL_SPLITK_TC)
            aux = cfg.get("tma_burst", 1)
            r = (kind, M, N, K, r[4], cfg["split_k"], cfg["stages"], 0, aux, cfg.get("ahead", 0),
                 cfg.get("reducers", 0), us_alone[key], 2 * N * K / us_alone[key] / 1e3)
        out.append(r)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out-inc", default=INC)
    ap.add_argument("--out-log", default=None)
    ap.add_argument("--rounds", type=int, default=40)
    ap.add_argument("--only-m", type=int, nargs="*", default=None,
                    help="tune only these M; the table's rows (and the log's entries) for other M are kept")
    ap.add_argument("--sequence", nargs="*", choices=sorted(SEQUENCES), default=None,
                    help="then refine these workloads' rows with their whole steps timed (sequence_refine)")
    ap.add_argument("--sequence-only", nargs="+", choices=sorted(SEQUENCES), default=None,
                    help="only refine these workloads' rows of the existing table in sequence (uses --out-log's "
                         "timings alone)")
    args = ap.parse_args(argv)
    if args.sequence_only:
        build.build()
        skg.load()
        torch.cuda.set_device(0)
        rows = [tuple(r) for r in read_rows(args.out_inc)]
        log = json.load(open(args.out_log or os.path.join(HERE, "csrc", "skg_plan_tune_log.json")))
        rows = sequence_refine(rows, log, tuple(args.sequence_only))
        write_table(args.out_inc, rows, None, 0.0)
        return
    kept_rows, kept_log = [], []
    if args.only_m:
        kept_rows = [r for r in read_rows(args.out_inc) if r[1] not in args.only_m]
        if args.out_log and os.path.exists(args.out_log):
            kept_log = [e for e in json.load(open(args.out_log)) if e["M"] not in args.only_m]
    build.build()
    skg.load()
    torch.cuda.set_device(0)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    rows, log = [], []
    t0 = time.time()
    for (N, K, epi), ms in shapes().items():
        wbytes = 2 * N * K
        copies = max(7, math.ceil(3 * l2 / wbytes))
        base = generate(Projection(64, N, K, epi, seed=900)).W.cuda()
        Ws = [base.roll(i, dims=0).contiguous() for i in range(copies)]   # distinct bytes, same statistics
        del base
        for M in ms:
            if args.only_m and M not in args.only_m:
                continue
            t = generate(Projection(M, N, K, epi, seed=901 + M))
            x = t.x.cuda()
            res = None if t.res is None else t.res.cuda()
            y = torch.empty(M, N, dtype=torch.float32 if epi == "fp32" else torch.bfloat16, device="cuda")
            results = []
            for cfg in candidates(M, N, K):
                us, info = time_config(M, N, K, epi, cfg, Ws, x, res, y, args.rounds)
                if us is not None:
                    results.append((us, cfg, info))
                    log.append({"M": M, "N": N, "K": K, "epilogue": epi, "config": cfg, "us": round(us, 3),
                                "weight_gbs": round(wbytes / us / 1e3, 1)})
            if M > 2:
                # reducers per tile, on the fastest launch shapes
                best = sorted(results, key=lambda r: r[0])[:REDUCER_SHAPES]
                for _, cfg0, info0 in best:
                    for r in (1, 2, 4, 8):
                        if r > cfg0["split_k"] or r == info0["reducers"]:
                            continue
                        cfg = dict(cfg0, reducers=r)
                        us, info = time_config(M, N, K, epi, cfg, Ws, x, res, y, args.rounds)
                        if us is not None:
                            results.append((us, cfg, info))
                            log.append({"M": M, "N": N, "K": K, "epilogue": epi, "config": cfg,
                                        "us": round(us, 3), "weight_gbs": round(wbytes / us / 1e3, 1)})
            us, cfg, info = min(results, key=lambda r: r[0])
            kind = info["kernel_kind"]
            rows.append((kind, M, N, K, skg.EPILOGUES[epi], info["split_k"],
                         info["stages"],
                         0, info["tma_burst"] if kind == skg.SKG_KERNEL_SPLITK_TC or
                         (info["split_k"] == 1 and info["stages"] >= 2) else 1,
                         cfg.get("ahead", 0), cfg.get("reducers", 0), us, wbytes / us / 1e3))
            print(f"N={N} K={K} {epi} M={M}: best {cfg} {us:.2f} us {wbytes / us / 1e3:.0f} GB/s", flush=True)
        del Ws
        torch.cuda.empty_cache()
    rows = sorted(kept_rows + rows, key=lambda r: (r[2], r[3], r[4], r[1]))
    log = kept_log + log
    if args.sequence:
        rows = sequence_refine(rows, log, tuple(args.sequence))
    write_table(args.out_inc, rows, args.out_log and log, time.time() - t0, args.out_log)
    print(f"wrote {args.out_inc} ({len(rows)} rows)")


def write_table(path, rows, log, seconds, log_path=None):
    """The table rows (and, given log_path, the timing log) as written by main."""
    with open(path, "w") as f:
        f.write("// skg_plan_table.inc -- measured picker table.\n//\n"
                "// Each row: { kernel_kind, M, N, K, epilogue, split_k, stages, grid, tma_burst, l2_ahead,\n"
                "// reducers } (reducers: CTAs of a split-K tile sharing its reduction, 0 = library default).\n"
                "// stages: TC ring stages / GEMV weight-ring slots per warp (0 = library default);\n"
                "// GEMV split 1: 0 = 16-byte loads into registers, 2 = one bulk copy per batch into\n"
                "// a shared-memory slot of the warp, whole rows per warp, 3 = the same batches in one\n"
                "// balanced wave (tma_burst = strips per copy for 2 and 3);\n"
                "// grid = 0 lets the library size the grid.  Written by projection_gemm_gb300/tune.py\n"
                f"// from back-to-back timings on {torch.cuda.get_device_name(0)} "
                f"({len(rows)} rows); the comment on each row is the\n"
                "// measured time per launch and weight-stream rate (launches of that row alone; the rows\n"
                "// of the batch sweep, the decode-layer chain and the wide and deep-K batches are then\n"
                "// chosen with their whole steps timed).\n")
        for r in rows:
            f.write("{%d, %d, %d, %d, %d, %d, %d, %d, %d, %d, %d},  // %.2f us, %.0f GB/s\n" % tuple(r[:13]))
    if log_path and log:
        with open(log_path, "w") as f:
            f.write("[\n" + ",\n".join(json.dumps(r) for r in log) + "\n]\n")


if __name__ == "__main__":
    main()
