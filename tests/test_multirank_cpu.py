"""The benchmark's multi-rank logic on CPU: two gloo ranks, no GPU.

Under torchrun every rank times its own batch (cells are independent, no
collective on the data path); the timed region is bracketed by barriers and the
reported time is the max over ranks. These tests run that code path with a step
whose cost differs by rank, and check the reference arm's rank-0-only rule.
"""
import io
import os
import socket
import sys
import time
from contextlib import redirect_stdout
from types import SimpleNamespace

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _SleepRunner:
    """A step that costs 2 ms x (rank + 1) of wall time and counts its calls."""

    def __init__(self, rank):
        self.rank = rank
        self.calls = []

    def step(self, i):
        time.sleep(0.002 * (self.rank + 1))
        self.calls.append(i)


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r = _SleepRunner(rank)
        ms = bench.time_steps(r, steps=6, warmup=3, world=world, timer=bench.HostTimer(), device="cpu")
        own = bench.max_over_ranks(1.0 + rank, world, "cpu")
        q.put((rank, ms, r.calls, own))
    finally:
        dist.destroy_process_group()


def test_timed_region_reports_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    for _ in procs:
        rank, ms, calls, own = q.get(timeout=120)
        out[rank] = (ms, calls, own)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert set(out) == {0, 1}
    ms0, calls0, own0 = out[0]
    ms1, calls1, own1 = out[1]
    # both ranks report the same time: the max over ranks
    assert ms0 == ms1
    # rank 1 sleeps 4 ms per step, so the max is at least that per step
    assert ms0 >= 4.0
    # exactly W warm-up steps then K timed steps, indices continuing
    assert calls0 == list(range(9)) and calls1 == list(range(9))
    assert own0 == own1 == 2.0


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    r = _SleepRunner(0)
    ms = bench.time_steps(r, steps=2, warmup=3, world=1, timer=bench.HostTimer(), device="cpu")
    assert ms >= 2.0 and r.calls == list(range(5))
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = SimpleNamespace(workload="cfg3", steps=1, warmup=3, ref_seconds_per_step=1.0)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) is None
    assert buf.getvalue() == ""


def test_gpus_flag_starts_one_rank_per_gpu():
    """`bench.py --gpus 2` outside torchrun starts two ranks itself (torch.distributed.run on
    127.0.0.1); the launcher self-test runs the same launch, timing and reporting path on CPU
    ranks, so the line must say n_gpus 2 and carry the slower rank's time."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_PORT")}
    env["OMP_NUM_THREADS"] = "1"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--launch-selftest",
                        "--steps", "5", "--warmup", "3"], capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["selftest"] is True and line["n_gpus"] == 2
    # rank 1 sleeps 4 ms a step: the reported time is the max over ranks
    assert line["ms_per_step"] >= 4.0
