"""pa_decode_attention_static: the entry point that allocates nothing.

It serves callers that have no way to allocate device memory.  One example
is a plugin inside another runtime that is handed only its input and output
buffers and may not call cudaMalloc, because the host runtime owns all
device memory.  Another is a serving loop that cannot afford the device
synchronisation a cudaMalloc may cause.  The entry point keeps its scratch
(task list and split partials) in a fixed 16 MiB array inside the library.

These tests call it through the C ABI twice in a row, each time with a plan
that splits sequences so the scratch array really carries partial results.
Each output is checked against the float64 oracle and against the regular
pa_decode_attention (caller workspace) on the same inputs, within the parity
tolerance.  A call must leave the device's memory use unchanged, and plans
too big for the array must be refused.  The file is named so that pytest
collects it last; it also passes on its own in a fresh process.
"""

from __future__ import annotations

import ctypes

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


def _regular(dd, plan):
    out = torch.empty_like(dd.q)
    ws = binding.alloc_workspace(plan, dd.device)
    binding.upload(plan, ws)
    binding.decode(dd.shape, plan, dd.q, dd.k_pages, dd.v_pages, dd.block_table, dd.seq_lens,
                   dd.w.scale, out, ws, dd.status)
    torch.cuda.synchronize()
    return out


def test_static_entry_point_matches_oracle_and_regular_twice(lib):
    w = workloads.make_custom(seq_lens=[1500, 37, 700, 1, 4000], num_q_heads=16, num_kv_heads=4,
                              head_dim=128, seed=4242)
    dd = DeviceDecode(w)
    dd.append()
    torch.cuda.synchronize()
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
    plans = [binding.Plan(dd.shape, w.seq_lens, dd.num_sms, 0),
             binding.Plan(dd.shape, w.seq_lens, dd.num_sms, 5)]
    for plan in plans:
        assert plan.c.num_groups > 0              # partials go through the scratch array
        assert plan.workspace_bytes <= binding.STATIC_WORKSPACE_BYTES
    for call, plan in enumerate(plans):           # two calls in a row
        regular = _regular(dd, plan)
        got = torch.full_like(dd.q, float("nan"))
        dd.status.zero_()
        binding.decode_static(dd.shape, plan, dd.q, dd.k_pages, dd.v_pages, dd.block_table,
                              dd.seq_lens, w.scale, got, dd.status)
        torch.cuda.synchronize()
        assert int(dd.status.item()) == 0, f"call {call}: device status {int(dd.status.item()):#x}"
        g = got.cpu().numpy().astype(np.float64)
        assert_close(g, want, f"static call {call} against the oracle")
        assert_close(g, regular.cpu().numpy().astype(np.float64), f"static call {call} against "
                     "pa_decode_attention")


def test_static_entry_point_allocates_nothing(lib):
    """Once a first call has loaded the library's device code, a call leaves
    torch's allocator and the device's free memory exactly as they were."""
    w = workloads.make_custom(seq_lens=[3000, 64, 900], num_q_heads=8, num_kv_heads=2,
                              head_dim=128, seed=4343)
    dd = DeviceDecode(w)
    dd.append()
    plan = binding.Plan(dd.shape, w.seq_lens, dd.num_sms, 4)
    out = torch.empty_like(dd.q)

    def call():
        binding.decode_static(dd.shape, plan, dd.q, dd.k_pages, dd.v_pages, dd.block_table,
                              dd.seq_lens, w.scale, out, dd.status)
        torch.cuda.synchronize()
    call()
    before = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info())
    for _ in range(3):
        call()
    after = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info())
    assert after == before
    assert int(dd.status.item()) == 0


def test_static_entry_point_rejects_oversized_plan(lib):
    # 2048 sequences x 8 KV heads x 2 splits: the partials alone exceed 16 MiB
    lens = np.full(2048, 64, np.int32)
    shape = binding.make_shape(2048, 32, 8, 128, 16, 4, 2048 * 4)
    plan = binding.Plan(shape, lens, 152, 2)
    assert plan.workspace_bytes > binding.STATIC_WORKSPACE_BYTES
    fake = ctypes.c_void_p(0x10000)   # never touched: the size check comes first
    code = lib.pa_decode_attention_static(ctypes.byref(shape), ctypes.byref(plan.c), fake, fake,
                                          fake, fake, fake, ctypes.c_float(0.1), fake, fake, None)
    assert code == 3, binding.STATUS_NAMES.get(code, code)
