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


def test_reference_arm_prints_the_contract_line(capsys, monkeypatch):
    """bench.py --impl reference times the CPU oracle and prints one JSON line
    with the keys the benchmark contract asks for."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    rc = bench.main(["--impl", "reference", "--workload", "decode_T8", "--steps", "2", "--warmup", "3",
                     "--cpu-seconds", "0.05"])
    assert rc == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3 and d["gpu_launches"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "T=8" in d["config"]["workload"]
