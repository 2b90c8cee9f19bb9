"""Failure detection on the device: every wait of the split-decode and
multi-token kernels is bounded, and a wait that runs out is reported, not
trapped.

A plan made with wait_limit_ns = 1 (plan options) gives each wait for a page
copy (or, in the tcgen05 kernel, for an MMA or another warp) one nanosecond:
far less than a copy takes, so the waits give up while the copies they wait
for still land.  Then, for each kernel:
  - the call returns and the stream completes (the context stays usable);
  - *dev_status is exactly PA_DEV_TIMEOUT, no other bit;
  - every output the gave-up tasks feed is left as it was (a NaN sentinel
    here), and every other output is the oracle's;
  - a fresh plan upload with the default limit gives the oracle's answer
    everywhere (a gave-up call may leave split counters non-zero, which the
    upload resets).
No copy is left unissued or broken: only the waiting gives up early.
"""

from __future__ import annotations

import zlib

import numpy as np
import pytest

import oracle
from paged_kv_decode_24_gb300 import binding, workloads
from paged_kv_decode_24_gb300.runner import DeviceDecode
from tests.cache8 import oracle_append_decode
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

SHORT_NS = 1


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


def split_rows(got, want, what, dtype="fp16"):
    """Each (token, head) row is untouched (all NaN) or the oracle's; returns
    how many rows were untouched."""
    g = got.astype(np.float64)
    nan_any, nan_all = np.isnan(g).any(axis=-1), np.isnan(g).all(axis=-1)
    assert np.array_equal(nan_any, nan_all), f"{what}: a row was partly written"
    done = ~nan_all
    if done.any():
        assert_close(g[done], want[done], f"{what}: rows that completed", dtype=dtype)
    return int(nan_all.sum())


def lens_for(n, seed):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(1, 1600, n)]


DECODE = [
    # (name, Hq, Hkv, kv, merge)
    ("mha_cuda_cores", 8, 8, "fp16", "split"),
    ("gqa4_tensor_cores", 16, 4, "fp16", "split"),
    ("gqa4_combine_kernel", 16, 4, "fp16", "combine"),
    ("int8_cache", 16, 4, "int8", "split"),
    ("fp8_cache", 16, 4, "fp8", "split"),
]


@pytest.mark.parametrize("case", DECODE, ids=[c[0] for c in DECODE])
def test_decode_wait_limit_runs_out(case):
    name, hq, hkv, kv, merge = case
    lens = lens_for(40, zlib.crc32(name.encode()))
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                              seed=zlib.crc32(name.encode()) ^ 5, kv=kv, forced_splits=0)
    dd = DeviceDecode(w)
    if kv in ("int8", "fp8"):
        dd.append8()
        want, _ = oracle_append_decode(w)
        call = dd.decode8
    else:
        dd.append()
        kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                  w.seq_lens)
        want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
        call = dd.decode
    torch.cuda.synchronize()
    untouched_total = 0
    for _ in range(3):
        # several splits per sequence, so split tasks and their merge are in
        # play; a call that timed out may leave split counters non-zero, so
        # each call gets its own upload, as the header asks
        dd.make_plan(forced_splits=3, merge=merge, wait_limit_ns=SHORT_NS)
        assert dd.plan_obj.c.wait_limit_ns == SHORT_NS and dd.plan_obj.c.num_groups > 0
        out = torch.full_like(dd.q, float("nan"))
        dd.status.zero_()
        call(out=out)
        status = dd.read_status()      # synchronises: the call has completed
        assert status == binding.PA_DEV_TIMEOUT, f"{name}: status {status:#x}"
        untouched_total += split_rows(out.float().cpu().numpy(), want, name)
    assert untouched_total > 0, f"{name}: no task gave up"
    # a fresh upload with the default limit: every output is the oracle's
    dd.make_plan(forced_splits=3, merge=merge)
    out = torch.full_like(dd.q, float("nan"))
    dd.status.zero_()
    call(out=out)
    assert dd.read_status() == 0
    assert_close(out.float().cpu().numpy(), want, f"{name} after a fresh upload")


@pytest.mark.parametrize("rows", [128, 64], ids=["tcgen05", "mma_sync"])
def test_prefill_wait_limit_runs_out(rows):
    lens = [900, 1500, 333, 64, 1200, 700]
    qls = [300, 128, 333, 10, 600, 1]
    w = workloads.make_custom(seq_lens=lens, num_q_heads=16, num_kv_heads=4, head_dim=128,
                              seed=4711 + rows, q_lens=qls)
    kp, vp = oracle.kv_append_tokens(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                     w.seq_lens, w.q_lens)
    want = oracle.prefill_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.q_lens, w.scale)
    dd = DeviceDecode(w)
    dd.make_prefill_plan(rows_per_tile=rows, wait_limit_ns=SHORT_NS)
    assert dd.pf_plan.c.wait_limit_ns == SHORT_NS
    dd.append_tokens()
    untouched = 0
    for _ in range(3):
        out = torch.full_like(dd.q, float("nan"))
        dd.status.zero_()
        dd.prefill(out=out)
        status = dd.read_status()
        assert status == binding.PA_DEV_TIMEOUT, f"rows={rows}: status {status:#x}"
        untouched += split_rows(out.float().cpu().numpy(), want, f"prefill rows={rows}")
    assert untouched > 0
    dd.make_prefill_plan(rows_per_tile=rows)
    out = torch.full_like(dd.q, float("nan"))
    dd.status.zero_()
    dd.prefill(out=out)
    assert dd.read_status() == 0
    assert_close(out.float().cpu().numpy(), want, f"prefill rows={rows} after a fresh plan")
