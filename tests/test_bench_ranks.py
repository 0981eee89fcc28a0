"""bench.py's multi-rank host logic, on CPU with world-size-2 gloo groups.

The decode path shards as independent replicas: every rank runs the same
per-GPU workload, the job's time is the slowest rank's, and the whole-job
rate counts the units of all ranks.  These tests run that logic (rank
environment, max over ranks, whole-job rate) in two gloo processes, and check
that the reference arm runs on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, w, local = bench.rank_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    per_rank_ms = 10.0 + 5.0 * r          # rank 1 is the slower one
    job_ms = bench.max_over_ranks(per_rank_ms, dist, "cpu")
    rate = bench.job_rate(w, 32769, job_ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "job_ms": job_ms, "rate": rate}, f)


def test_max_over_ranks_and_job_rate_gloo(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert (d["rank"], d["world"], d["local"]) == (r, 2, r)
        assert d["job_ms"] == 15.0                      # the slowest rank's time, on every rank
        assert d["rate"] == pytest.approx(2 * 32769 / 15e-3)


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    old = dict(os.environ)
    try:
        os.environ.clear()
        os.environ.update(env)
        assert bench.rank_env() == (0, 1, 0)
    finally:
        os.environ.clear()
        os.environ.update(old)
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_rate(1, 1000, 2.0) == pytest.approx(5e5)


def _run_reference(rank, world, extra=()):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--gpus", str(world), "--workload", "0", "--steps", "2", "--warmup", "1",
                           *extra], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_silently():
    p = _run_reference(1, 2)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    p = _run_reference(0, 2)
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_step_launch_counts_follow_the_documented_forms():
    # bench.py's gpu_launches claim: the kernels one vq_decode_step launches on
    # each workload, per include/vqattn.h (fused append: 2; the 1.5-bit format
    # with its sliced scan: 3; more pairs than SMs: 3)
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    got = {i: bench.step_launches(W.WORKLOADS[i], 152) for i in (1, 2, 3, 4, 5)}
    assert got == {1: 2, 2: 2, 3: 2, 4: 3, 5: 3}
    # a 1.5-bit batch with more (sequence, KV head) pairs than SMs: scan, merge, attention, merge
    w = W.custom(batch=64, num_q_heads=32, num_kv_heads=8, k_sub=8, k_bits=12, v_sub=8, v_bits=12)
    assert bench.step_launches(w, 152) == 4
