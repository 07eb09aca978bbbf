"""The multi-process host path of bench.py (replicas only: barrier and max of the
timings over ranks) on the CPU with gloo at world size 2."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench

    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    q.put((rank, d.max(1.5 * (rank + 1), "cpu")))
    d.barrier()
    d.close()


def test_replica_reduction_with_gloo():
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
    assert got == [(0, 3.0), (1, 3.0)]


def test_single_process_needs_no_process_group():
    import bench

    d = bench.Dist()
    assert d.world in (1, int(os.environ.get("WORLD_SIZE", "1")))
    if d.world == 1:
        d.init("gloo")
        assert d.pg is None and d.max(2.5, "cpu") == 2.5
