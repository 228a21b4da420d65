"""The N > 1 launch path of bench.py on CPU: two ranks over gloo on
127.0.0.1.  The attention path shards into independent problems (replicas),
so the only cross-rank operations are the barrier and the max-over-ranks of
the timings; the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import bench, torch.distributed as dist
world, rank, local = bench.dist_setup(want_cuda=False)
assert world == 2 and dist.get_world_size() == 2 and rank == dist.get_rank()
bench.barrier(world)
# max over ranks of rank-dependent timings: both ranks see the larger one
m = bench.max_over_ranks(1.5 + rank, world)
assert m == 2.5, m
print("rank", rank, "ok", flush=True)
dist.destroy_process_group()
"""


def test_two_gloo_ranks_barrier_and_max():
    port = free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e[-2000:]
    assert sorted(o.strip() for o, _ in outs) == ["rank 0 ok", "rank 1 ok"]


def test_reference_arm_under_torchrun_prints_one_line():
    """bench.py --impl reference launched like the driver does for N = 2:
    rank 0 times the oracle and prints one JSON line, rank 1 exits 0."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "3", "--warmup", "3", "--ref-rows", "8"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
