"""Host logic of the multi-process benchmark on CPU ranks (gloo, world size 2).

`bench.py --gpus N` runs N independent replicas (the path has no exchange
step); the job's time is the slowest rank's time and the throughput counts
every rank's units. The reference arm runs on rank 0 only.
"""

import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_RANK_SCRIPT = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
rank, _, world = bench.dist_env()
dist.init_process_group("gloo", init_method="env://")
local_ms = 10.0 + 5.0 * rank                      # rank 1 is the slower replica
job_ms = bench.world_max(local_ms, world)
value = bench.job_throughput(1000, world, 4, job_ms)
dist.barrier()
dist.destroy_process_group()
print(json.dumps({{"rank": rank, "job_ms": job_ms, "value": value}}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(script, world, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", script], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_world_max_and_job_throughput_over_two_gloo_ranks():
    import json
    outs = _launch(_RANK_SCRIPT.format(root=ROOT), 2)
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for r in res:
        assert r["job_ms"] == pytest.approx(15.0)                 # the slower rank's time
        assert r["value"] == pytest.approx(1000 * 2 * 4 / 0.015)  # both ranks' units


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.world_max(7.5, 1) == 7.5
    assert bench.job_throughput(32768, 1, 10, 1000.0) == pytest.approx(327680.0)


def test_reference_arm_runs_on_rank_zero_only():
    script = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench\n"
              "class A: steps = 1; warmup = 0; gpus = 2\n"
              "rc = bench.reference_arm(A()); print('rc', rc)\n")
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, "-c", script], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "rc 0"                            # no JSON line, no oracle work
