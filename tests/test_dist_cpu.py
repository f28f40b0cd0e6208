"""The N > 1 path of bench.py on CPU: two gloo ranks.

The op has no exchange step; bench.py runs one independent replica per rank
and uses torch.distributed only for the barrier around the timed region and
for the max of the per-rank times.  This checks that logic with world size 2
(gloo, 127.0.0.1) without a GPU.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    got = d.max(10.0 * (rank + 1))
    d.barrier()
    d.close()
    q.put((rank, d.world, got))


def test_two_rank_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=10) for _ in range(2))
    assert results == [(0, 2, 20.0), (1, 2, 20.0)]


def test_single_process_needs_no_process_group(monkeypatch):
    for key in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(key, raising=False)
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init("gloo")
    assert d.world == 1 and d.pg is None
    assert d.max(3.5) == 3.5
    d.barrier()
    d.close()
