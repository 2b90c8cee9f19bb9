"""Two decode calls in flight at once on two streams, each with its own
workspace, status word and output: the library keeps no per-call state
outside the caller's buffers, so each result matches the oracle."""

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


def test_two_streams_in_flight():
    cases = [([700, 33, 1024, 5], 32, 8, 128, 0), ([2048], 32, 32, 128, 16)]
    runs = []
    for case in cases:
        lens, hq, hkv, d, splits = case
        w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                  seed=zlib.crc32(str(case).encode()) ^ 11, forced_splits=splits)
        dd = DeviceDecode(w)
        dd.make_plan()
        runs.append((w, dd, torch.cuda.Stream()))
    torch.cuda.synchronize()
    for _ in range(20):   # interleave the two streams' launches
        for w, dd, s in runs:
            with torch.cuda.stream(s):
                binding.append_decode(dd.shape, dd.plan_obj, dd.q, dd.k_new, dd.v_new, dd.k_pages,
                                      dd.v_pages, dd.block_table, dd.seq_lens, w.scale, dd.out,
                                      dd.workspace, dd.status)
    torch.cuda.synchronize()
    for w, dd, _ in runs:
        assert int(dd.status.item()) == 0
        kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                  w.seq_lens)
        want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
        assert_close(dd.out.cpu().numpy(), want, "two streams")
