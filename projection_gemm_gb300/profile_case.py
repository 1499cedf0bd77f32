"""Run one projection a few times through the C ABI -- a small, fixed workload
for profilers (ncu captures of a single kernel launch).

usage: python -m projection_gemm_gb300.profile_case M N K [epilogue] [launches]
The operands are the seeded synthetic tensors of `inputs.py` (seed 11); the
default plan is used; the process exits non-zero on any library error.
"""
import sys

import torch

from . import build, skg
from .inputs import Projection, generate


def main(argv):
    M, N, K = int(argv[0]), int(argv[1]), int(argv[2])
    epi = argv[3] if len(argv) > 3 else "bf16"
    launches = int(argv[4]) if len(argv) > 4 else 3
    build.build()
    skg.load()
    torch.cuda.set_device(0)
    t = generate(Projection(M, N, K, epi, seed=11))
    x, W = t.x.cuda(), t.W.cuda()
    res = None if t.res is None else t.res.cuda()
    y = torch.empty(M, N, dtype=torch.float32 if epi == "fp32" else torch.bfloat16, device="cuda")
    plan = skg.Plan(M, N, K, epi)
    print(plan.info())
    for _ in range(launches):
        plan.run(x, W, res, y)
    torch.cuda.synchronize()
    plan.check()
    plan.close()
    print("ok")


if __name__ == "__main__":
    main(sys.argv[1:])
