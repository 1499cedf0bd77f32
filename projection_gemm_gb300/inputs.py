"""Seeded synthetic inputs for the skinny decode projection.

This module only draws random numbers and lays them out; it does none of the
projection's arithmetic.  The test suite hands the same bits to the CUDA
library and to the CPU oracle, and the benchmark uses the same recipe.

Recipe (stated here once, used everywhere):
  * ``numpy.random.SeedSequence(seed).spawn(4)`` gives one child sequence
    each for x [M,K], W [N,K], residual [M,N] and the outlier-row choice;
    a tensor is cut into 64 row blocks (fewer if it has fewer rows), block i
    is filled with float32 standard normals by ``Generator(PCG64(child_i))``
    where child_i is the i-th of ``child.spawn(blocks)``; the blocks are
    filled by a thread pool, and the result does not depend on its size;
  * x ~ N(0, 1), W ~ N(0, 1/K) (standard deviation 1/sqrt(K)), residual
    ~ N(0, var) with the variance given per workload (1 or 4);
  * each draw is cast to bfloat16 with round-to-nearest-even;
  * outlier channels: floor(N/100) distinct rows of W, picked by
    ``permutation(N)[:N//100]`` after W is drawn, are multiplied by 16 in
    bf16, which is exact (a power of two).

The pages that describe the method measure a production model
("Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly",
experimental setup and results); no weights or activations of that model are
available, so these synthetic tensors with the projection shapes of a decode
layer stand in for them.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Projection:
    """One projection problem: y[M,N] = x[M,K] . W[N,K]^T (+ residual)."""
    M: int
    N: int
    K: int
    epilogue: str = "bf16"          # "bf16", "bf16_residual" or "fp32"
    seed: int = 0
    residual_var: float = 1.0       # variance of the residual draw
    outlier_frac: float = 0.0       # 0.01: 1% of W rows scaled by 16
    name: str = ""

    @property
    def has_residual(self) -> bool:
        return self.epilogue == "bf16_residual"

    @property
    def out_bytes_per_elem(self) -> int:
        return 4 if self.epilogue == "fp32" else 2

    def weight_bytes(self) -> int:
        return 2 * self.N * self.K

    def algorithmic_bytes(self) -> int:
        """W + x + residual (if any) + y, each touched once."""
        b = 2 * self.N * self.K + 2 * self.M * self.K
        if self.has_residual:
            b += 2 * self.M * self.N
        return b + self.out_bytes_per_elem * self.M * self.N

    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


@dataclasses.dataclass
class Tensors:
    x: torch.Tensor                 # bf16 [M,K], CPU
    W: torch.Tensor                 # bf16 [N,K], CPU
    res: Optional[torch.Tensor]     # bf16 [M,N], CPU, or None
    outlier_rows: Optional[torch.Tensor]


_BLOCKS = 64


def _fill(job):
    seq, out = job
    np.random.Generator(np.random.PCG64(seq)).standard_normal(out.shape, dtype=np.float32, out=out)


def _normal_bf16(seq: np.random.SeedSequence, shape, std: float) -> torch.Tensor:
    rows = shape[0]
    f = np.empty(shape, dtype=np.float32)
    nb = max(1, min(_BLOCKS, rows))
    bounds = [rows * i // nb for i in range(nb + 1)]
    jobs = [(c, f[bounds[i]:bounds[i + 1]]) for i, c in enumerate(seq.spawn(nb))]
    if f.size >= (1 << 20):
        with cf.ThreadPoolExecutor(max_workers=min(nb, os.cpu_count() or 1)) as ex:
            list(ex.map(_fill, jobs))
    else:
        for j in jobs:
            _fill(j)
    if std != 1.0:
        f *= np.float32(std)
    return torch.from_numpy(f).to(torch.bfloat16)


def generate(p: Projection, with_weight: bool = True) -> Tensors:
    """Draw the tensors of ``p`` (CPU, bf16) following the module recipe."""
    sx, sw, sr, so = np.random.SeedSequence(int(p.seed)).spawn(4)
    x = _normal_bf16(sx, (p.M, p.K), 1.0)
    W = _normal_bf16(sw, (p.N, p.K), 1.0 / math.sqrt(p.K)) if with_weight else None
    res = _normal_bf16(sr, (p.M, p.N), math.sqrt(p.residual_var)) if p.has_residual else None
    rows = None
    if p.outlier_frac > 0 and W is not None:
        count = int(p.N * p.outlier_frac)
        perm = np.random.Generator(np.random.PCG64(so)).permutation(p.N)
        rows = torch.from_numpy(perm[:count].astype(np.int64))
        W[rows] = W[rows] * 16
    return Tensors(x=x, W=W, res=res, outlier_rows=rows)


def bits(t: torch.Tensor):
    """Raw uint16 bit patterns (numpy) of a CPU bf16 tensor."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


# --------------------------------------------------------------------------
# The workloads.  Shapes are those of a decode layer's projections; the
# pages give none, so these are the shapes the method is measured on here.
# --------------------------------------------------------------------------
SWEEP_M = (1, 2, 4, 8, 16, 32, 64)
WIDE_M = (1, 2, 8, 32, 64)
DEEPK_M = (1, 4, 16, 64)
CHAIN_M = (1, 8, 64)

# (K, N, epilogue) of the five back-to-back projections of one decode layer.
CHAIN_STAGES: Tuple[Tuple[int, int, str], ...] = (
    (7168, 12288, "bf16"),           # wide input projection
    (8192, 7168, "bf16_residual"),   # output projection + residual
    (7168, 384, "fp32"),             # router-score GEMM, fp32 out
    (7168, 4096, "bf16"),            # latent input projection
    (4096, 7168, "bf16_residual"),   # projection back + residual
)


def pr1() -> Projection:
    """M=1, K=N=1024, + residual ~N(0,1), seed 0."""
    return Projection(1, 1024, 1024, "bf16_residual", seed=0, residual_var=1.0,
                      name="pr1")


def sweep(M: int, seed: Optional[int] = None) -> Projection:
    """Batch sweep: K=N=7168, no residual; default seed = index of M."""
    s = SWEEP_M.index(M) if seed is None else seed
    return Projection(M, 7168, 7168, "bf16", seed=s, name=f"sweep_m{M}")


def wide(M: int) -> Projection:
    """Wide input projection: K=7168, N=12288, 1% outlier rows x16."""
    return Projection(M, 12288, 7168, "bf16", seed=100 + WIDE_M.index(M),
                      outlier_frac=0.01, name=f"wide_m{M}")


def deepk(M: int) -> Projection:
    """Deep-K output projection: K=16384, N=7168, residual ~N(0,4)."""
    return Projection(M, 7168, 16384, "bf16_residual", seed=200 + DEEPK_M.index(M),
                      residual_var=4.0, name=f"deepk_m{M}")


def chain(M: int) -> List[Projection]:
    """The five projections of the decode-layer chain at batch M."""
    out = []
    for i, (K, N, epi) in enumerate(CHAIN_STAGES):
        out.append(Projection(M, N, K, epi, seed=300 + 10 * CHAIN_M.index(M) + i,
                              residual_var=1.0, name=f"chain_m{M}_s{i}"))
    return out


def all_workloads() -> Dict[str, List[Projection]]:
    return {
        "pr1": [pr1()],
        "sweep": [sweep(m) for m in SWEEP_M],
        "wide": [wide(m) for m in WIDE_M],
        "deepk": [deepk(m) for m in DEEPK_M],
        "chain": [p for m in CHAIN_M for p in chain(m)],
    }
