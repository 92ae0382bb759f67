"""Host logic of bench.py's multi-GPU (replicas) path on CPU: two gloo ranks
reduce their timings with MAX and compute the whole-job rate; the reference
arm runs on rank 0 only."""
import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = 10.0 + 5.0 * rank                     # rank 1 is the slow replica
    ms_max = bench.max_over_ranks(ms_local, dist, "cpu")
    rate = bench.job_rate(1e12, 4, world, ms_max)
    dist.barrier()
    dist.destroy_process_group()
    out_q.put((rank, ms_max, rate))


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, rate in res:
        assert ms_max == 15.0
        assert rate == pytest.approx(1e12 * 4 * 2 / 15e-3)


def test_reference_arm_runs_on_rank_zero_only():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
           "--warmup", "0", "--ref-sample-tokens", "32", "--workload", "tiny_t256_e8"]
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env["RANK"] = "0"
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["unit"] == "TFLOPS" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
