"""The bench's N>1 path on the CPU: two gloo ranks, each a replica of the workload.

The path has no exchange step on one GPU (every head is local), so ranks are
independent replicas; the only cross-rank operation is the max-reduce of the timed
region, and the whole-job value is all ranks' work over the slowest rank's time.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 if rank == 0 else 250.0   # rank 1 is the slow one
        per_s, total_ms = bench.replica_throughput(local_ms, 1000.0, world)
        q.put((rank, per_s, total_ms))
    finally:
        dist.destroy_process_group()


def test_replica_throughput_max_reduces_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, per_s, total_ms in got:
        assert total_ms == 250.0                        # the slowest rank's time
        assert abs(per_s - 2 * 1000.0 / 0.25) < 1e-6    # both ranks' units over it


def test_replica_throughput_single_rank():
    sys.path.insert(0, ROOT)
    import bench

    per_s, total_ms = bench.replica_throughput(50.0, 10.0, 1)
    assert total_ms == 50.0 and abs(per_s - 200.0) < 1e-9


def test_reference_arm_prints_one_line_on_cpu():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1", "--ref-rows", "16"], capture_output=True, text=True,
                       env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    import json

    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, env=env, timeout=300,
                       cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""
