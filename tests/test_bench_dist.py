"""bench.py's multi-rank host logic on CPU: two gloo ranks (the timing takes the slowest
rank, the value counts every rank's tokens) and the reference arm's idle non-zero ranks."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import os, sys, json
sys.path.insert(0, os.environ["GDN_ROOT"])
import torch, torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank = dist.get_rank()
ms = bench._max_over_ranks(dist, 1.0 + 2.0 * rank, torch.device("cpu"))
value = bench._job_value(64 * 10, dist.get_world_size(), ms)
dist.barrier()
dist.destroy_process_group()
print(json.dumps({"rank": rank, "ms": ms, "value": value}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r), WORLD_SIZE="2",
                   LOCAL_RANK=str(r), GDN_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            pytest.fail("gloo ranks did not finish")
        assert p.returncode == 0, err
        outs.append(out.strip().splitlines()[-1])
    import json
    res = sorted((json.loads(o) for o in outs), key=lambda d: d["rank"])
    assert [d["ms"] for d in res] == [3.0, 3.0]  # rank 1 took 3 ms: the job took 3 ms
    assert all(d["value"] == pytest.approx(64 * 10 * 2 / 3e-3) for d in res)


def test_job_value_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(None, 2.5, None) == 2.5
    assert bench._job_value(64 * 256, 1, 12.8) == pytest.approx(64 * 256 / 12.8e-3)


def test_reference_arm_rank1_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
