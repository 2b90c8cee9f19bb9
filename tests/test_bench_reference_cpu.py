"""The benchmark's reference arm on CPU: `bench.py --impl reference` times
the float64 oracle on the host cores and prints one JSON line with the
primary arm's metric, unit and workload, a cpu_baseline that describes the
run, and an e2e block with no host-device bytes."""

from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "1",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference"
    assert d["metric"].startswith("decode-attention")
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"].startswith("tiny paged decode")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_default_is_the_headline_workload():
    """With no --config the line is about workload 4 (LLaMA-3-8B heads, batch
    160), and its config dict is exactly the one the GPU arm prints, so the
    two lines compare like for like."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_decode_24_gb300 import workloads
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["config"]["config_id"] == 4 and d["config"]["batch"] == 160
    args = argparse.Namespace(config=4, kv="fp16", dtype="fp16")
    assert d["config"] == bench.workload_config(args, workloads.make_config(4), 1)
