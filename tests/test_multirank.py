"""The N > 1 path of bench.py on the CPU, as two gloo ranks (the multi-GPU
layout is replicas over trees: no collective touches the data path, only the
timing barrier and the max-over-ranks reduction of the elapsed time)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys
import torch
import torch.distributed as dist
sys.path.insert(0, sys.argv[1])
import bench
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
out = {"ms": ms, "seeds": bench.rank_seeds(rank, 4), "value": bench.whole_job_value(world, 4, ms)}
dist.barrier()
with open(os.path.join(sys.argv[2], "r%d.json" % rank), "w") as f:
    json.dump(out, f)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_report_the_slowest_rank(tmp_path):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT, ROOT, str(tmp_path)],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
    r0 = json.load(open(tmp_path / "r0.json"))
    r1 = json.load(open(tmp_path / "r1.json"))
    assert r0["ms"] == r1["ms"] == 15.0                       # the slower rank's time
    assert not set(r0["seeds"]) & set(r1["seeds"])            # disjoint trees per rank
    assert r0["value"] == r1["value"] == pytest.approx(2 * 4 / 15e-3)  # whole-job trees per second


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
