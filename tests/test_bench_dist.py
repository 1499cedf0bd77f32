"""The multi-rank side of bench.py on CPU: two gloo ranks (spawned
processes) aggregate like a 2-GPU run does -- the slowest rank's time and the
sum of both ranks' units."""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t, u = bench.aggregate(1.5 + rank, 100.0 * (rank + 1), world)
    q.put((rank, t, u, bench.dist_env()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_max_time_and_sums_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u, env in got:
        assert t == 2.5 and u == 300.0
        assert env == (rank, 2, 0)
