"""Run one projection a few times through the C ABI -- a small, fixed workload
for profilers (ncu captures of a single kernel launch).

usage: python -m projection_gemm_gb300.profile_case M N K [epilogue] [launches]
                                                    [--kind gemv|tc] [--split S] [--stages D] [--burst B]
       python -m projection_gemm_gb300.profile_case M --chain-group [--independent] [launches]
The operands are the seeded synthetic tensors of `inputs.py` (seed 11); the
default plan is used unless --kind (skg_plan_force_kernel) or --split /
--stages / --burst (skg_plan_force) force a configuration.  --chain-group runs the five decode-layer chain
projections at M as one group launch (skg_group, each projection ordered
after the previous one, or with --independent in no order) instead.  The
process exits non-zero on any library error.
"""
import argparse
import sys

import torch

from . import build, skg
from .inputs import Projection, generate


def chain_group(M, launches, ordered=True):
    from .inputs import CHAIN_STAGES
    ts = [generate(Projection(M, N, K, epi, seed=11 + i)) for i, (K, N, epi) in enumerate(CHAIN_STAGES)]
    xs = [t.x.cuda() for t in ts]
    Ws = [t.W.cuda() for t in ts]
    rs = [None if t.res is None else t.res.cuda() for t in ts]
    ys = [torch.empty(M, N, dtype=torch.float32 if epi == "fp32" else torch.bfloat16, device="cuda")
          for (K, N, epi) in CHAIN_STAGES]
    g = skg.Group(M, [N for _, N, _ in CHAIN_STAGES], [K for K, _, _ in CHAIN_STAGES],
                  [e for _, _, e in CHAIN_STAGES], [0, 1, 1, 1, 1] if ordered else None)
    print(g.info())
    for _ in range(launches):
        g.run(xs, Ws, rs, ys)
    torch.cuda.synchronize()
    g.check()
    g.close()
    print("ok")


def main(argv):
    if "--chain-group" in argv:
        rest = [a for a in argv if a not in ("--chain-group", "--independent")]
        build.build()
        skg.load()
        torch.cuda.set_device(0)
        chain_group(int(rest[0]), int(rest[1]) if len(rest) > 1 else 3, "--independent" not in argv)
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("M", type=int)
    ap.add_argument("N", type=int)
    ap.add_argument("K", type=int)
    ap.add_argument("epilogue", nargs="?", default="bf16")
    ap.add_argument("launches", nargs="?", type=int, default=3)
    ap.add_argument("--kind", choices=("gemv", "tc"), default=None)
    ap.add_argument("--split", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--burst", type=int, default=0)
    a = ap.parse_args(argv)
    M, N, K, epi, launches = a.M, a.N, a.K, a.epilogue, a.launches
    build.build()
    skg.load()
    torch.cuda.set_device(0)
    t = generate(Projection(M, N, K, epi, seed=11))
    x, W = t.x.cuda(), t.W.cuda()
    res = None if t.res is None else t.res.cuda()
    y = torch.empty(M, N, dtype=torch.float32 if epi == "fp32" else torch.bfloat16, device="cuda")
    plan = skg.Plan(M, N, K, epi)
    if a.kind:
        plan.force_kernel(skg.SKG_KERNEL_GEMV if a.kind == "gemv" else skg.SKG_KERNEL_SPLITK_TC)
    if a.split or a.stages or a.burst:
        plan.force(split_k=a.split, stages=a.stages, tma_burst=a.burst)
    print(plan.info())
    for _ in range(launches):
        plan.run(x, W, res, y)
    torch.cuda.synchronize()
    plan.check()
    plan.close()
    print("ok")


if __name__ == "__main__":
    main(sys.argv[1:])
