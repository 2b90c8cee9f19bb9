"""The C ABI inside a captured CUDA graph: pa_plan_upload and
pa_decode_attention captured once, replayed after the inputs and the staged
plan have changed.  A graph reads the buffers as they are at replay, and a
plan rewritten into the same pinned staging buffer with the same structure
keeps the captured upload valid.
"""

from __future__ import annotations

import zlib

import numpy as np
import pytest

import oracle
from paged_kv_decode_24_gb300 import binding, workloads
from paged_kv_decode_24_gb300.runner import DeviceDecode
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


def oracle_decode(w, q):
    return oracle.decode_attention(q, w.k_pages, w.v_pages, w.block_table, w.seq_lens, w.scale)


@pytest.mark.parametrize("case", [([300, 129, 1000, 5], 32, 8, 128, 0),
                                  ([4096], 32, 32, 128, 16)])
def test_captured_graph_replays_with_new_inputs_and_plan(case):
    lens, hq, hkv, d, splits = case
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              seed=zlib.crc32(str(case).encode()) ^ 5, forced_splits=splits)
    dd = DeviceDecode(w)
    lens_host = np.ascontiguousarray(w.seq_lens)
    probe = binding.Plan(dd.shape, lens_host, dd.num_sms, w.forced_splits)
    staging = torch.empty(int(probe.c.blob_bytes), dtype=torch.uint8).pin_memory()
    plan = binding.Plan(dd.shape, lens_host, dd.num_sms, w.forced_splits, host_buffer=staging)
    ws = binding.alloc_workspace(plan, dd.device)
    # one eager call first: the kernels' one-time setup happens outside capture
    binding.upload(plan, ws)
    binding.decode(dd.shape, plan, dd.q, dd.k_pages, dd.v_pages, dd.block_table, dd.seq_lens,
                   w.scale, dd.out, ws, dd.status)
    torch.cuda.synchronize()
    dd.out.zero_()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        binding.upload(plan, ws)
        binding.decode(dd.shape, plan, dd.q, dd.k_pages, dd.v_pages, dd.block_table,
                       dd.seq_lens, w.scale, dd.out, ws, dd.status)

    g.replay()
    torch.cuda.synchronize()
    assert int(dd.status.item()) == 0
    assert_close(dd.out.cpu().numpy(), oracle_decode(w, w.q), f"graph replay 1 {case}")

    # new q in place, and the plan made again into the same staging buffer
    rng = np.random.default_rng(17)
    q2 = rng.normal(0.0, 0.5, size=w.q.shape).astype(np.float16)
    dd.q.copy_(torch.from_numpy(q2).to(dd.device))
    plan2 = binding.Plan(dd.shape, lens_host, dd.num_sms, w.forced_splits, host_buffer=staging)
    assert plan2.structure() == plan.structure()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert int(dd.status.item()) == 0
    assert_close(dd.out.cpu().numpy(), oracle_decode(w, q2), f"graph replay 2 {case}")
