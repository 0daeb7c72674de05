"""bench.py's multi-rank plumbing on CPU (gloo, world size 2): the barrier,
the max over ranks, and rank-0-only output of the reference arm."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist = bench.init_dist(world, "gloo")
    cpu = torch.device("cpu")
    bench.barrier(dist, cpu)
    m = bench.max_over_ranks(dist, 10.0 * (rank + 1), cpu)
    bench.barrier(dist, cpu)
    q.put((rank, m, bench.dist_env()))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[1] for g in got] == [20.0, 20.0]
    assert [g[2][:2] for g in got] == [(0, 2), (1, 2)]


def test_reference_arm_is_silent_on_other_ranks(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_warmup_below_three_is_refused():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.main(["--warmup", "2"]) == 2
