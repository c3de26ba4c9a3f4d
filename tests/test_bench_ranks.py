"""The benchmark's multi-rank host logic on the CPU (gloo, world size 2): the
path has no cross-rank exchange, so N GPUs run independent replicas; the job
value is every rank's tokens over the slowest rank's time, and the reference
arm runs on rank 0 only."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [10.0, 25.0][rank]
    value, job_ms = bench.job_value(local_ms, 1000, 4, world, dist, "cpu")
    q.put((rank, value, job_ms))
    dist.destroy_process_group()


def test_job_value_is_total_tokens_over_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, value, job_ms in res:
        assert job_ms == 25.0                      # the slowest rank's time, on every rank
        assert abs(value - 2 * 1000 * 4 / 0.025) < 1e-6


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", ADALN_SKIP_BUILD="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "1", "--gpus", "2"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
