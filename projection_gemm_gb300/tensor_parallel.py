"""Tensor-parallel projections across ranks: the host side.

"Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly" describes two
ways the decode projections are spread over GPUs:

* method details 2 "Overlap computation and communication": the output
  projection is row-parallel -- its reduction dimension K is split across
  GPUs, every GPU computes a partial result, and the partials are summed
  (all-reduce) with the attention residual added in the same step;
* method details 3: the router-score GEMM and the latent input projection,
  which read the same hidden state, are computed as one GEMM whose output
  columns are distributed over the GPUs, and the slices are exchanged.

Row-parallel (``RowParallelProjection``): rank r of R owns canonical K chunks
[16r/R, 16(r+1)/R), i.e. columns [rK/R, (r+1)K/R) of x and W.  ``skg_run`` of
a plan set to that shard (``skg_plan_set_k_shard``) leaves the rank's fp32
partial -- the value of its subtree of the canonical reduction tree; the
partials are all-gathered in rank order and ``skg_combine_partials`` adds the
top levels of the tree, the residual and the one rounding, so every rank ends
with exactly the bits of a single launch over the whole K.

Column-parallel (``ColumnParallelGroup``): rank r owns rows [rN/R, (r+1)N/R)
of every weight of a group of projections that share x; one group launch
(``skg_group``, no ordering between its projections) computes the rank's
slices and an all-gather assembles every output.  A row of y depends only on
its own row of W, so the slices have the bits of the unsharded launch.

The exchange uses ``torch.distributed`` (NCCL between GPUs, gloo between CPU
processes); this module only moves bytes and calls the library -- every
arithmetic step runs in the library's kernels.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

from . import skg

RANKS = (1, 2, 4, 8)


def k_shard_columns(K: int, rank: int, ranks: int) -> Tuple[int, int]:
    """Columns [c0, c1) of x and W that rank `rank` of `ranks` owns in a
    row-parallel projection (whole canonical chunks: K % 1024 == 0)."""
    if ranks not in RANKS or not 0 <= rank < ranks:
        raise ValueError(f"rank {rank} of {ranks}: ranks must be one of {RANKS}")
    if ranks > 1 and K % (skg.CANONICAL_CHUNKS * 64) != 0:
        raise ValueError(f"K={K}: a K split needs K % {skg.CANONICAL_CHUNKS * 64} == 0")
    w = K // ranks
    return rank * w, (rank + 1) * w


def n_shard_rows(N: int, rank: int, ranks: int) -> Tuple[int, int]:
    """Rows [n0, n1) of W (columns of y) that rank `rank` owns in a
    column-parallel projection: contiguous, sizes differing by at most one."""
    if ranks < 1 or not 0 <= rank < ranks:
        raise ValueError(f"rank {rank} of {ranks}")
    return rank * N // ranks, (rank + 1) * N // ranks


def all_gather(t, group=None) -> List:
    """All ranks' tensors of t's shape, in rank order (torch.distributed)."""
    import torch
    import torch.distributed as dist
    out = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(out, t.contiguous(), group=group)
    return out


class RowParallelProjection:
    """y = x.W^T (+ residual) with K split across the ranks of a group."""

    def __init__(self, M: int, N: int, K: int, epilogue: str, rank: int, ranks: int):
        self.M, self.N, self.K = M, N, K
        self.epilogue, self.rank, self.ranks = epilogue, rank, ranks
        self.columns = k_shard_columns(K, rank, ranks)
        self.plan = skg.Plan(M, N, K, "fp32")
        self.plan.set_k_shard(rank, ranks)

    def partial(self, x_shard, W_shard, out, stream=None):
        """This rank's fp32 partial [M, N] of x_shard [M, K/R] and W_shard [N, K/R]."""
        self.plan.run(x_shard, W_shard, None, out, stream)
        return out

    def combine(self, partials: Sequence, residual, y, stream=None):
        """y from all ranks' partials (rank order), on this rank's device."""
        skg.skg_combine_partials(self.M, self.N, list(partials), residual, y, self.epilogue, stream)
        return y

    def run(self, x_shard, W_shard, residual, y, partial, group=None, stream=None):
        """partial -> all-gather -> combine: every rank ends with the whole y."""
        self.partial(x_shard, W_shard, partial, stream)
        return self.combine(all_gather(partial, group), residual, y, stream)

    def close(self):
        self.plan.close()


class ColumnParallelGroup:
    """Projections that read the same x (e.g. router scores and the latent
    input projection), each weight's rows split across the ranks: one group
    launch per rank, then an all-gather of every output's slices."""

    def __init__(self, M: int, N: Sequence[int], K: int, epilogues: Sequence[str], rank: int, ranks: int):
        self.M, self.N, self.K = M, list(N), K
        self.rows = [n_shard_rows(n, rank, ranks) for n in self.N]
        self.group = skg.Group(M, [n1 - n0 for n0, n1 in self.rows], [K] * len(self.N), list(epilogues), None)

    def run_local(self, x, W_slices, y_slices, stream=None):
        """This rank's slices: W_slices[i] = W_i[n0:n1] (contiguous rows)."""
        self.group.run([x] * len(self.N), W_slices, None, y_slices, stream)
        return y_slices

    def gather(self, y_slices, group=None) -> List:
        """Every output whole, from all ranks' slices (equal slice sizes)."""
        import torch
        outs = []
        for ys in y_slices:
            parts = all_gather(ys, group)
            outs.append(torch.cat(parts, dim=1))
        return outs

    def close(self):
        self.group.close()
