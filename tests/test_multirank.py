"""The multi-rank bench logic on CPU with gloo, world size 2.

Decode attention shards by sequence with no exchange, so more GPUs run independent
replicas: the job's time is the slowest rank's (max over ranks) and its throughput
counts every rank's bytes.  The reference arm runs on rank 0 only.
"""
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
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    ms = [0.20, 0.35][rank]
    got = bench.max_over_ranks(ms)
    gbs = bench.whole_job_gbs(1_000_000_000, world, got)
    q.put((rank, got, gbs))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, got, gbs in res:
        assert got == 0.35                     # both ranks see the slowest rank's time
        assert abs(gbs - 2 * 1.0 / 0.35e-3) < 1e-6 * gbs   # 2 replicas x 1 GB in 0.35 ms


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=120, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.whole_job_gbs(2_000_000_000, 1, 1.0) == 2000.0
