"""The multi-process host logic of bench.py on CPU: world size 2 over gloo.

Under torchrun every rank runs its own replica layers (weak scaling, no
collective on the data path); the only collectives are the barrier around the
timed region, the max of the ranks' times and the sum of their bytes.  The
reference arm runs on rank 0 alone.  These tests run those steps with two
CPU processes."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import bench
ws, rank, local = bench.dist_env()
dist = bench.dist_init(ws, "gloo")
# each rank: its own (elapsed ms, bytes moved)
ms = [10.0, 14.0][rank]
nbytes = [1.0e9, 3.0e9][rank]
bench.barrier(dist)
ms_max = bench.max_over_ranks(ms, dist)
total = bench.sum_over_ranks(nbytes, dist)
steps_max = int(bench.max_over_ranks(float([20, 35][rank]), dist))
bench.barrier(dist)
print(json.dumps({"rank": rank, "ws": ws, "ms_max": ms_max, "total": total, "steps": steps_max,
                  "value": total / (ms_max * 1e-3) / 1e9}))
dist.destroy_process_group()
"""


def run_ranks(code: str, args=(), ws: int = 2, timeout: float = 120.0):
    port = free_port()
    procs = []
    for r in range(ws):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(ws),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", code, ROOT, *args], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, e
        outs.append(o)
    return outs


def test_weak_scaling_aggregation_two_ranks():
    outs = run_ranks(WORKER)
    recs = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for r in recs:
        assert r["ws"] == 2
        assert r["ms_max"] == 14.0              # the slowest rank's time
        assert r["total"] == 4.0e9              # every rank's bytes
        assert r["steps"] == 35                 # ranks agree on the step count
        assert abs(r["value"] - 4.0e9 / 14e-3 / 1e9) < 1e-9


REF = r"""
import sys, json
sys.path.insert(0, sys.argv[1])
import bench
sys.argv = ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
            "--workload", "tiny", "--cpu-seconds", "1"]
rc = bench.main()
sys.exit(rc or 0)
"""


def test_reference_arm_runs_on_rank_zero_only():
    outs = run_ranks(REF, timeout=600.0)
    lines0 = [l for l in outs[0].splitlines() if l.startswith("{")]
    lines1 = [l for l in outs[1].splitlines() if l.startswith("{")]
    assert len(lines0) == 1 and not lines1
    rec = json.loads(lines0[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
