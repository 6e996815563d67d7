"""The benchmark's multi-rank host logic with two gloo ranks on CPU: the
timing aggregation takes the slowest rank, the job throughput counts every
rank's bytes, and the reference arm runs on rank 0 only.  (The library path
itself is replicas only: no data-path collective.)"""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ws, r, _ = bench.dist_env()
    assert (ws, r) == (world, rank)
    bench.dist_barrier(ws)
    slowest = bench.dist_max(10.0 + rank * 5.0, ws)  # rank 1 is 5 ms slower
    out.put((rank, slowest, bench.job_gbs(1e9, ws, 100, slowest)))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_and_job_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29000 + os.getpid() % 2000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, gbs in got:
        assert slowest == 15.0                      # max over ranks
        assert gbs == pytest.approx(2 * 1e9 * 100 / 15e-3 / 1e9)  # both ranks' bytes / slowest time


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
