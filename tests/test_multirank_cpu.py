"""Multi-rank host logic of bench.py on CPU: two gloo ranks (world_size 2).

Rows are independent, so N GPUs run N replicas of the step with no collective in the data path;
the only cross-rank traffic is the timing barrier and the max over ranks of the elapsed time.
These tests run that logic with the gloo backend on the host, and check that under torchrun
the reference arm prints one line from rank 0 while the other rank exits cleanly.
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


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
world, rank, local = bench.dist_setup()
assert world == 2
bench.barrier(world)
m = bench.max_over_ranks(world, float(10 + rank))
units = 1000 * world
print(json.dumps({{"rank": rank, "max": m, "value": units / m}}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def test_max_over_ranks_and_barrier_with_gloo(tmp_path):
    script = tmp_path / "w.py"
    script.write_text(WORKER.format(root=ROOT))
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(r), LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    assert all(r["max"] == 11.0 for r in res)          # max over ranks, seen by every rank
    assert all(abs(r["value"] - 2000 / 11.0) < 1e-9 for r in res)


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    p = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    doc = json.loads(lines[0])
    assert doc["impl"] == "reference" and doc["n_gpus"] == 2 and doc["value"] > 0
    assert doc["cpu_baseline"]["kind"] == "oracle"
    assert doc["e2e"]["h2d_bytes_per_step"] == 0
