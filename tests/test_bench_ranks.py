"""The multi-rank logic of bench.py on CPU: two gloo ranks (127.0.0.1).

bench.py under torchrun times the same workload on every rank, takes the slowest
rank's time per step and reports the whole job's matrices per second; the reference
arm runs on rank 0 only.  These are checked here without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


WORKER = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo", init_method="env://")
rank, world, _ = bench.dist_env()
ms = [2.0, 5.0][rank]
e2e = [7.0, 3.0][rank]
out = bench.max_over_ranks([ms, e2e])
print(json.dumps({{"rank": rank, "world": world, "max": out,
                  "rate": bench.whole_job_rate(10, world, out[0])}}), flush=True)
dist.barrier()
dist.destroy_process_group()
"""


def _run_two(code, extra_env=None):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   WORLD_SIZE="2", LOCAL_RANK=str(rank))
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=120)
        assert p.returncode == 0, e
        outs.append(o)
    return outs


def test_slowest_rank_sets_the_time_and_the_rate_counts_every_rank():
    outs = _run_two(WORKER.format(root=ROOT))
    for o in outs:
        d = json.loads(o.strip().splitlines()[-1])
        assert d["world"] == 2
        assert d["max"] == [5.0, 7.0]                       # element-wise max over the ranks
        assert d["rate"] == pytest.approx(10 * 2 / 5e-3)     # 20 matrices per 5 ms


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.whole_job_rate(7, 1, 3.5) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only():
    code = f"""
import sys
sys.path.insert(0, {ROOT!r})
import bench
class A: workload = "single"; steps = 1; warmup = 3
bench.run_reference(A())
"""
    port = _free_port()
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK="1", WORLD_SIZE="2",
               LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""                           # rank 1: no work, no line
    env["RANK"], env["LOCAL_RANK"] = "0", "0"
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
