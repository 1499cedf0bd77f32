"""The exchange side of the tensor-parallel projections on CPU ranks: two
gloo processes, each with its own K columns or N rows, all-gather their
pieces in rank order (the same calls move fp32 partials and output slices
between GPUs over NCCL)."""
import multiprocessing as mp
import os
import socket

import pytest
import torch


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from projection_gemm_gb300 import tensor_parallel as tp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        M, N, K = 4, 300, 8192
        c0, c1 = tp.k_shard_columns(K, rank, world)
        part = torch.full((M, N), float(rank + 1), dtype=torch.float32) + torch.arange(N, dtype=torch.float32)
        got = tp.all_gather(part)
        n0, n1 = tp.n_shard_rows(N, rank, world)
        ys = torch.full((M, n1 - n0), float(10 * rank), dtype=torch.float32)
        cat = torch.cat(tp.all_gather(ys), dim=1)
        q.put((rank, (c0, c1), [float(g[0, 0]) for g in got], (n0, n1), cat[0].tolist()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gather_partials_and_slices_in_rank_order():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, cols0, got0, rows0, cat0), (r1, cols1, got1, rows1, cat1) = res
    assert cols0 == (0, 4096) and cols1 == (4096, 8192)
    assert got0 == got1 == [1.0, 2.0]                    # rank 0's partial first
    assert rows0 == (0, 150) and rows1 == (150, 300)
    assert cat0 == cat1 == [0.0] * 150 + [10.0] * 150


def test_shard_bounds():
    from projection_gemm_gb300 import tensor_parallel as tp
    assert [tp.k_shard_columns(7168, r, 4) for r in range(4)] == [(0, 1792), (1792, 3584), (3584, 5376),
                                                                 (5376, 7168)]
    assert tp.k_shard_columns(1000, 0, 1) == (0, 1000)
    for bad in ((1000, 0, 2), (8192, 2, 2), (8192, 0, 3)):
        with pytest.raises(ValueError):
            tp.k_shard_columns(*bad)
    rows = [tp.n_shard_rows(4480, r, 8) for r in range(8)]
    assert rows[0][0] == 0 and rows[-1][1] == 4480 and all(a[1] == b[0] for a, b in zip(rows, rows[1:]))
