"""GPU: the README's Python example runs as written and its output matches
the float64 oracle.  The example's code block is read from README.md and
executed with a small seeded workload's tensors bound to its names."""

from __future__ import annotations

import os
import re

import numpy as np
import pytest

import oracle
from paged_kv_decode_24_gb300 import workloads
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


def test_readme_python_example():
    text = open(os.path.join(ROOT, "README.md"), encoding="utf-8").read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) == 1
    w = workloads.make_custom(seq_lens=[300, 37, 1025], num_q_heads=8, num_kv_heads=2,
                              head_dim=128, seed=91)

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    env = {"q": dev(w.q), "k_pages": dev(w.k_pages), "v_pages": dev(w.v_pages),
           "block_table": dev(w.block_table), "seq_lens": dev(w.seq_lens),
           "k_new": dev(w.k_new), "v_new": dev(w.v_new), "D": w.head_dim}
    exec(compile(blocks[0], "README.md", "exec"), env)
    torch.cuda.synchronize()
    assert int(env["status"].item()) == 0
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
    assert abs(w.scale - w.head_dim ** -0.5) < 1e-12
    assert_close(env["out"].cpu().numpy(), want, "README example")
