"""CPU tests of bench.py's multi-process path (world size 2, gloo): the
rendezvous from the torchrun environment, the barrier, the max over ranks
that every timing goes through, and the reference arm's rank-0-only rule.
The data path has no collective (replicas), so these are the only
cross-rank steps."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    ws, r, local = bench.dist_setup()
    try:
        assert dist.get_backend() == "gloo"
        bench.barrier(ws)
        # every rank's own elapsed time goes in; the slowest rank's comes out
        t = bench.max_over_ranks(ws, 1.5 + 2.0 * r)
        # the reference arm: only rank 0 works and prints
        class A:
            workload, steps, warmup, gpus = "w4_tiny", 1, 0, world
        rc = bench.run_reference(A, ws, r) if r != 0 else 0
        bench.barrier(ws)
        q.put((r, ws, local, t, rc))
    finally:
        dist.destroy_process_group()


def test_two_rank_barrier_and_max_over_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == world for g in got)
    assert [g[2] for g in got] == [0, 1]
    assert all(g[3] == 3.5 for g in got)   # max(1.5, 3.5) on both ranks
    assert got[1][4] == 0                  # rank 1 of the reference arm exits 0 without work


def test_single_process_needs_no_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup() == (1, 0, 0)
    assert bench.max_over_ranks(1, 2.25) == 2.25
    bench.barrier(1)
