"""GPU parity at the long end: one 131072-token sequence (four times the
longest benchmark context) beside a short one, on each split kernel (CUDA
cores for MHA, tensor cores for GQA, the INT8 cache), with the automatic
plan aimed at two waves of resident CTAs (plan option waves = 2).  The
planner cuts the long sequence into well over a hundred splits, so the split
merge combines that many partials per head.  Every head of both sequences is
compared with the float64 oracle.
"""

from __future__ import annotations

import pytest

import oracle
from paged_kv_decode_24_gb300 import workloads
from paged_kv_decode_24_gb300.runner import DeviceDecode
from tests.cache8 import oracle_append_decode
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


LONG = 131072


@pytest.mark.parametrize("hq,hkv,kv", [(8, 8, "fp16"), (16, 2, "fp16"), (8, 2, "int8"),
                                       (8, 8, "fp8")])
def test_131072_token_context(hq, hkv, kv):
    w = workloads.make_custom(seq_lens=[LONG, 77], num_q_heads=hq, num_kv_heads=hkv,
                              head_dim=128, seed=8000 + hq + hkv, kv=kv)
    dd = DeviceDecode(w)
    dd.make_plan(waves=2)
    assert dd.plan_obj.c.max_splits >= 100
    if kv in ("int8", "fp8"):
        dd.append8()
        got = dd.decode8().cpu().numpy()
    else:
        dd.append()
        got = dd.decode().cpu().numpy()
    assert dd.read_status() == 0
    if kv in ("int8", "fp8"):
        want, _ = oracle_append_decode(w)
    else:
        kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                  w.seq_lens)
        want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
    assert_close(got, want, f"{kv} Hq={hq} Hkv={hkv}, every head")
