"""The multi-GPU bench path on CPU: ranks are independent replicas joined only
for timing (max over ranks) and output (rank 0 prints), exercised with the
gloo backend and world size 2."""
import json
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


SCRIPT = textwrap.dedent("""
    import json, os, sys
    import torch.distributed as dist
    sys.path.insert(0, %r)
    import bench
    dist.init_process_group("gloo")
    rank, world = dist.get_rank(), dist.get_world_size()
    # per-rank step times differ; bench.py's own aggregation must report the
    # slowest rank and the tokens of all ranks
    ms = bench.max_over_ranks(1.0 + rank, world, "cpu")
    value = bench.job_value(world, 64, ms)
    if rank == 0:
        print(json.dumps({"world": world, "ms": ms, "value": value}))
    dist.destroy_process_group()
""")


def test_two_rank_replica_aggregation(tmp_path):
    script = tmp_path / "agg.py"
    script.write_text(SCRIPT % ROOT)
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", str(script)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=240, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1                              # rank 0 alone prints
    out = json.loads(lines[0])
    assert out["world"] == 2 and out["ms"] == 2.0       # max over ranks
    assert out["value"] == pytest.approx(2 * 64 / 2e-3)


def test_reference_arm_two_ranks_rank0_only(tmp_path):
    # bench.py --impl reference under torchrun: rank 0 runs the CPU oracle and
    # prints one line; the other rank exits 0 without work
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3", "--gpus", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["value"] > 0 and out["cpu_baseline"]["kind"] == "oracle"
