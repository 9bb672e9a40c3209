"""The N>1 host path of bench.py on CPU: two gloo ranks (replicas only, no
data-path collective).  The barrier and the max over ranks are the only
cross-rank steps; the reported value counts the work of every rank over the
slowest rank's time, and the reference arm runs on rank 0 alone."""

import json
import os
import socket
import subprocess
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_PROGRAM = r"""
import json, os, sys
sys.path.insert(0, os.getcwd())
import bench
world, rank, local = bench.dist_env()
d = bench.Dist(world)
d.barrier()
slowest = d.max(10.0 * (rank + 1))          # rank r took 10 (r + 1) ms
value = bench.replica_value(world, 1e9, slowest)
d.barrier()
d.close()
print(json.dumps({"rank": rank, "local": local, "max_ms": slowest, "value": value}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                   RANK=str(rank), LOCAL_RANK=str(rank))
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_PROGRAM], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=120)
            assert p.returncode == 0, err[-2000:]
            outs.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["local"] == o["rank"]
        assert o["max_ms"] == 20.0                      # the slower rank's time on both
        assert o["value"] == pytest.approx(2 * 1e9 / 20e-3 / 1e9)  # both ranks' units


def test_replica_value_is_weak_scaling():
    import bench
    one = bench.replica_value(1, 134246400 * 28, 0.75)
    assert bench.replica_value(4, 134246400 * 28, 0.75) == pytest.approx(4 * one)
    assert bench.replica_value(2, 1e9, 10.0) == pytest.approx(200.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = types.SimpleNamespace(gpus=2, steps=1, warmup=3)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""   # no line and no oracle work on rank 1
