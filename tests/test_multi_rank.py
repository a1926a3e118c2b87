"""The N > 1 host path of bench.py on CPU (gloo, world size 2).

The forward shards into independent (sequence, head) replicas with no data
exchange, so the only multi-rank logic is host-side: every rank times its
replica, the job takes the slowest rank's time (an all-reduce of the maximum),
and the throughput counts every rank's tokens.  The reference arm runs on rank
0 alone; the other ranks exit without work.
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
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, "cpu")
        out[rank] = (ms, bench.whole_job_rate(ms, world, 16384))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    world = 2
    times = [1.25, 1.5]
    out = mp.Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), times, out), nprocs=world, start_method="spawn")
    for r in range(world):
        ms, rate = out[r]
        assert ms == 1.5
        assert rate == pytest.approx(world * 16384 / 1.5e-3)


def test_single_rank_keeps_its_own_time():
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.whole_job_rate(2.0, 1, 1000) == pytest.approx(5e5)


def test_reference_arm_runs_on_rank_zero_only():
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
        procs.append(subprocess.Popen(
            [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
             "--steps", "1", "--warmup", "3", "--gpus", "2"],
            cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=600) for p in procs]
    assert [p.returncode for p in procs] == [0, 0], [o[1][-2000:] for o in outs]
    lines0 = [ln for ln in outs[0][0].splitlines() if ln.startswith("{")]
    lines1 = [ln for ln in outs[1][0].splitlines() if ln.startswith("{")]
    assert len(lines0) == 1 and lines1 == []
    line = json.loads(lines0[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle"
