"""The benchmark's multi-replica path on CPU: two gloo ranks.

bench.py --gpus N runs N independent replicas (the path needs no exchange);
the only cross-rank steps are the barrier around the timed region and the
max over ranks of the step time.  These run here with the gloo backend.
"""

from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, sys.argv[1])
import bench
rank = int(os.environ["RANK"])
world, r, local = bench.dist_setup(None)
assert (world, r) == (2, rank)
bench.barrier(world)
mine = [3.0, 5.0][rank]
worst = bench.max_over_ranks(mine, world, "cpu")
value = bench.job_value(1_000_000_000, worst, world)
import torch.distributed as dist
dist.destroy_process_group()
print(json.dumps({"rank": rank, "worst": worst, "value": value}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code, extra_env=None):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code, ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_two_gloo_ranks_take_the_slowest_step():
    import json
    outs = _launch(WORKER)
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for r in res:
        assert r["worst"] == 5.0                      # max over ranks
        assert r["value"] == pytest.approx(2 * 1e9 / 5e-3 / 1e9)   # two replicas' bytes


def test_reference_arm_prints_on_rank_zero_only():
    code = r"""
import os, sys
sys.path.insert(0, sys.argv[1])
sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3", "--config", "1"]
import bench
bench.main()
"""
    outs = _launch(code)
    assert outs[1].strip() == ""
    import json
    line = json.loads(outs[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
