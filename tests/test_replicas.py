"""The multi-GPU form of the bench is N independent replicas (the path has no
exchange step): a gloo barrier around the timed region and the max of the
ranks' step times. This runs that host logic with two CPU ranks over gloo."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=2)
    ws, r, local = bench.dist_env()
    bench.dist_barrier(ws)
    ms = bench.dist_max(1.0 + r, ws)   # rank 1 is the slower replica
    bench.dist_barrier(ws)
    q.put((r, ws, local, ms, bench.replica_value(ws, 1.0e12, ms)))
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_the_whole_job():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    for r, ws, local, ms, value in res:
        assert ws == 2 and local == r
        assert ms == 2.0                                   # max over ranks
        assert value == pytest.approx(2 * 1.0e12 / 2.0e-3 / 1e12)   # both replicas' work over the slowest time
