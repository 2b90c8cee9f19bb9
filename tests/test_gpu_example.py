"""GPU: the Python usage example (examples/decode_step.py) runs as shipped
and its output matches the float64 oracle."""

from __future__ import annotations

import importlib.util
import os

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


def test_decode_step_example():
    spec = importlib.util.spec_from_file_location(
        "decode_step", os.path.join(ROOT, "examples", "decode_step.py"))
    ex = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(ex)
    w = workloads.make_custom(seq_lens=[300, 37, 1025], num_q_heads=8, num_kv_heads=2,
                              head_dim=128, seed=91)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out, status = ex.decode_step(dev(w.q), dev(w.k_new), dev(w.v_new), dev(w.k_pages),
                                 dev(w.v_pages), dev(w.block_table), dev(w.seq_lens))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
    assert abs(w.scale - w.head_dim ** -0.5) < 1e-12
    assert_close(out.cpu().numpy(), want, "examples/decode_step.py")
