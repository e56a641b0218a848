"""The N>1 host logic of bench.py on CPU: two ranks over gloo.

The path runs replicas only (every GPU holds its own virtual mesh), so the
only cross-rank steps are the barrier and the max over ranks of the timed
region; the whole-job value is every rank's bytes over the slowest time.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        slowest = bench.reduce_over_ranks(dist, ms, torch.device("cpu"), "max")
        total = bench.reduce_over_ranks(dist, 1.0e9, torch.device("cpu"), "sum")
        out[rank] = (slowest, total, bench.whole_job_gbs(1.0e9, world, slowest))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        slowest, total, gbs = res[r]
        assert slowest == 15.0                       # every rank sees the slowest time
        assert total == 2.0e9
        assert gbs == pytest.approx(2.0e9 / 15e-3 / 1e9)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_over_ranks(None, 3.5, torch.device("cpu")) == 3.5
    assert bench.whole_job_gbs(6.0e9, 1, 1.0) == pytest.approx(6000.0)


def test_reference_arm_prints_once_under_torchrun():
    """`bench.py --impl reference` launched as 2 ranks: rank 0 alone times the
    oracle and prints one JSON line; the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
