"""GPU: the Python usage examples (examples/decode_step.py,
examples/serving_loop.py) run as shipped and their outputs match the float64
oracle."""

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


def test_serving_loop_example():
    """examples/serving_loop.py: after steps with page allocation, a swap-out
    and a new sequence, every layer's last-step output matches the oracle
    over the final pools, the swapped pages came back bit for bit, and the
    allocator holds exactly the pages no sequence uses."""
    spec = importlib.util.spec_from_file_location(
        "serving_loop", os.path.join(ROOT, "examples", "serving_loop.py"))
    ex = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(ex)
    r = ex.serve()
    table, lens = r["block_table"], r["seq_lens"]
    used = table[table >= 0]
    assert len(np.unique(used)) == len(used)               # no page in two rows
    assert r["free"] == r["k_pages"][0].shape[0] - len(used)
    assert all((table[b] >= 0).sum() == -(-int(L) // ex.PAGE) for b, L in enumerate(lens))
    host_k, host_v, pages, (dev_k, dev_v) = r["swapped"]
    assert torch.equal(host_k, dev_k) and torch.equal(host_v, dev_v)
    for layer, out in enumerate(r["out"]):
        want = oracle.decode_attention(r["q"][layer].cpu().numpy(),
                                       r["k_pages"][layer].cpu().numpy(),
                                       r["v_pages"][layer].cpu().numpy(), table, lens, r["scale"])
        assert_close(out.cpu().numpy(), want, f"examples/serving_loop.py layer {layer}")
