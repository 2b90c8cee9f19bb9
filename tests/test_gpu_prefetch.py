"""The L2 prefetch that the split-decode kernels issue before waiting on the
previous kernel, at its widest setting: every CTA and all 32 lanes of every
warp prefetch, so every block-table entry a warp owns goes through the
bounds checks.  The knobs are read once per process, so the cases run in a
child process with the environment set.  Results must match the oracle as
with the default setting, and a block-table entry outside the pool must be
flagged and skipped, not prefetched.
"""

from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, zlib
sys.path.insert(0, sys.argv[1])
import numpy as np
import oracle
from paged_kv_decode_24_gb300 import binding, workloads
from paged_kv_decode_24_gb300.runner import DeviceDecode
from tests.parity import assert_close

def oracle_step(w):
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    return oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)

for case in [([5, 300, 129, 1000], 32, 8, 128, 0), ([96, 97, 1500], 16, 16, 128, 7),
             ([2000, 3, 640], 4, 4, 64, 0)]:
    lens, hq, hkv, d, splits = case
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              seed=zlib.crc32(str(case).encode()) ^ 7, forced_splits=splits)
    dd = DeviceDecode(w)
    dd.append()
    dd.make_plan(forced_splits=splits)
    got = dd.decode().cpu().numpy()
    assert dd.read_status() == 0, dd.read_status()
    assert_close(got, oracle_step(w), "prefetch " + str(case))

# INT8 cache
w = workloads.make_custom(seq_lens=[700, 33, 1024], num_q_heads=32, num_kv_heads=8, head_dim=128,
                          seed=71, kv="int8")
dd = DeviceDecode(w)
dd.make_plan()
dd.append_q8()
got = dd.decode_q8().cpu().numpy()
assert dd.read_status() == 0
kc, vc, ks, vs = oracle.kv_append_q8(w.k_codes, w.v_codes, w.k_scales, w.v_scales, w.k_new,
                                     w.v_new, w.block_table, w.seq_lens)
want = oracle.decode_attention_q8(w.q, kc, vc, ks, vs, w.block_table, w.seq_lens, w.scale)
assert_close(got, want, "prefetch int8")

# an entry outside the pool: flagged, skipped, never prefetched
w = workloads.make_custom(seq_lens=[40, 400], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=72)
w.block_table[1, 3] = w.num_pages + 1000
dd = DeviceDecode(w)
dd.make_plan()
out = dd.decode().cpu().numpy()
assert dd.read_status() & binding.PA_DEV_BAD_PAGE
assert np.all(np.isfinite(out.astype(np.float32)))
print("prefetch ok")
"""


def test_widest_prefetch_matches_oracle():
    env = dict(os.environ)
    env["PA_L2_PREFETCH_PAGES"] = "32"
    env["PA_L2_PREFETCH_CTAS"] = "2147483647"
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "prefetch ok" in r.stdout
