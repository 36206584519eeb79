"""The multi-rank path of bench.py on CPU: world size 2 over gloo.

The block shards by tokens with replicated weights (replicas only: no data-path
collective).  bench.py's job time is the slowest rank's and its throughput
counts every rank's units; both are checked here with real processes.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.argv = ["bench.py"]
    import bench
    ms_local = 10.0 * (rank + 1)                 # rank 1 is the slow one
    ms = bench.max_over_ranks(ms_local, dist, "cpu")
    q.put((rank, ms, bench.job_throughput(1000, world, 5, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [20.0, 20.0]
    assert res[0][2] == pytest.approx(2 * 1000 * 5 / 0.020)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    sys.argv = ["bench.py"]
    import bench
    assert bench.max_over_ranks(7.5, None, "cpu") == 7.5
    assert bench.job_throughput(10, 1, 2, 1000.0) == 20.0
