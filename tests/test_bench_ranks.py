"""Multi-rank bench logic on CPU: two gloo ranks (127.0.0.1), no GPU.

Each rank of `bench.py --gpus N` runs the step on its own row slices on its
own GPU; the aggregate time is the slowest rank's, reduced with MAX over all
ranks, the reference arm prints from rank 0 only, and a --gpus that does not
match the launch's WORLD_SIZE is an error, not a silent one-GPU run."""
from __future__ import annotations

import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r is slow on op "a" when r is large, on op "b" when r is small
        got = bench.max_over_ranks({"a": 1.0 + rank, "b": 5.0 - rank, "c": 2.5}, world, "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    for r in range(2):
        assert res[r] == {"a": 2.0, "b": 5.0, "c": 2.5}


def test_max_over_ranks_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    v = {"decode": 0.047, "lmhead": 0.138}
    assert bench.max_over_ranks(v, 1, "cpu") == v


def test_reference_arm_prints_only_on_rank_zero():
    env = {**os.environ, "RANK": "1", "WORLD_SIZE": "2", "PYTHONPATH": ROOT}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--cpu-seconds", "0.2"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_gpus_flag_must_match_the_launch():
    env = {**os.environ, "RANK": "0", "WORLD_SIZE": "2", "PYTHONPATH": ROOT}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "3", "--impl", "reference",
                        "--cpu-seconds", "0.2"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "does not match WORLD_SIZE" in r.stderr
