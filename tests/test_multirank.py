"""The multi-rank host logic of the benchmark on CPU (world size 2, gloo, 127.0.0.1): every
rank runs an independent replica (the rows are independent; no collective on the data
path), the job time is the slowest rank's, the job value sums the ranks' bytes, and the
reference arm runs on rank 0 alone."""

from __future__ import annotations

import json
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


def _worker(rank: int, world: int, port: int, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    # rank r took 1 + r seconds on its step loop and 5 - r on its end-to-end loop
    got = bench.ranks_max([1.0 + rank, 5.0 - rank], dist, device="cpu")
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, got))


def test_slowest_rank_sets_the_time_and_ranks_add_up():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 5.0]
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas of 10 steps of 1e9 bytes in the slowest rank's 2 s: 10 GB/s for the job
    assert bench.job_value(10**9, 10, 2, 2.0) == 10.0
    assert bench.ranks_max([3.0], None) == [3.0]


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_gpu_count_must_match_the_ranks():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode != 0
    assert "needs 2 ranks" in (r.stderr + r.stdout)
