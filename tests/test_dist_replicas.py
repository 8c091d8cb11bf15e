"""The bench's multi-rank path on CPU: two gloo ranks run the same setup, max-over-
ranks timing and whole-job aggregation the GPU replicas use (one process per GPU,
no data-path collective; only the timing reduction crosses ranks), and the
reference arm prints from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["REPO"])
import bench
rank, world, local = bench.dist_setup(2)
ms = 1.0 + rank                       # rank 1 is the slower replica
bench.barrier(world)
value, ms_max = bench.replica_throughput(1_000_000, ms, world)
print(json.dumps({"rank": rank, "world": world, "value": value, "ms_max": ms_max}))
import torch.distributed as dist
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code_or_args, world=2, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE=str(world), LOCAL_RANK=str(r), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), REPO=ROOT, CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        cmd = [sys.executable, "-c", code_or_args] if isinstance(code_or_args, str) else \
            [sys.executable] + code_or_args
        procs.append(subprocess.Popen(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=240)
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_two_gloo_ranks_aggregate_over_the_slowest_replica():
    outs = _launch(WORKER)
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o in outs), key=lambda r: r["rank"])
    assert [r["rank"] for r in res] == [0, 1] and all(r["world"] == 2 for r in res)
    for r in res:
        assert r["ms_max"] == pytest.approx(2.0)
        # 2 ranks x 1 MB over the slower rank's 2 ms
        assert r["value"] == pytest.approx(2 * 1_000_000 / 2e-3 / 1e9)


def test_reference_arm_prints_from_rank_zero_only():
    outs = _launch(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"])
    lines = [[l for l in o.splitlines() if l.startswith("{")] for o in outs]
    assert len(lines[0]) == 1 and lines[1] == []
    line = json.loads(lines[0][0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
