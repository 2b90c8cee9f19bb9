"""GPU parity of the multi-token path (pa_kv_append_tokens and
pa_prefill_attention) against the float64 oracle, through the C ABI, at the
decode path's tolerance (tests/parity.py), on both kernels: tcgen05 with
128-row tiles (the default) and mma.sync with 64-row tiles (plan option
rows_per_tile = 64).  The benchmark workloads compare every output.
"""

from __future__ import annotations

import zlib

import numpy as np
import pytest

import oracle
from paged_kv_decode_24_gb300 import binding, workloads
from paged_kv_decode_24_gb300.runner import DeviceDecode, MixedStep
from tests import oracle_pool
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


def close(got, want, what, dtype="fp16"):
    return assert_close(got, want, what, dtype=dtype)


def oracle_step(w, rows=None):
    kp, vp = oracle.kv_append_tokens(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                     w.seq_lens, w.q_lens)
    return oracle.prefill_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.q_lens, w.scale,
                                    rows=rows), (kp, vp)


def gpu_step(w, rows_per_tile=0):
    dd = DeviceDecode(w)
    dd.make_prefill_plan(rows_per_tile=rows_per_tile)
    dd.append_tokens()
    out = dd.prefill()
    status = dd.read_status()
    assert status == 0, f"device status {status:#x}"
    return out.float().cpu().numpy(), dd


CASES = [
    # (seq_lens, q_lens, Hq, Hkv, D)
    ([37, 100], [37, 5], 4, 2, 64),
    ([1, 2, 15, 16, 17, 31, 33, 64], [1, 2, 15, 16, 1, 8, 33, 20], 8, 8, 128),   # G = 1
    ([300, 129, 1000], [64, 129, 200], 32, 8, 128),                              # G = 4
    ([777, 50], [100, 50], 16, 2, 128),                                          # G = 8
    ([513, 257], [70, 257], 8, 1, 64),                                           # G = 8, D = 64
    ([2000, 3, 640], [1, 3, 640], 4, 4, 64),                                     # G = 1, D = 64
    ([96, 300, 5], [96, 0, 5], 16, 8, 128),                                      # G = 2, empty
]


def _ids(c):
    return f"L{c[0][:3]}_q{c[1][:3]}_G{c[2] // c[3]}_D{c[4]}"


@pytest.mark.parametrize("rows", [128, 64], ids=["tcgen05", "mma_sync"])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_prefill_parity_full(case, dtype, rows):
    lens, qls, hq, hkv, d = case
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              seed=zlib.crc32(str(case).encode()) ^ 32, q_lens=qls, dtype=dtype)
    got, dd = gpu_step(w, rows_per_tile=rows)
    assert dd.pf_plan.c.rows_per_tile == rows
    want, (kp, _) = oracle_step(w)
    close(got, want, f"prefill {case} {dtype} rows={rows}", dtype=dtype)
    assert np.array_equal(dd.k_pages.float().cpu().numpy(), kp.astype(np.float32))


def test_prefill_poisoned_pool_never_read():
    """Rows no sequence owns hold NaN: a read past a query's span would show."""
    w = workloads.make_custom(seq_lens=[1, 17, 250, 33], num_q_heads=8, num_kv_heads=2,
                              head_dim=128, seed=91, q_lens=[1, 9, 70, 33], poison=True)
    got, _ = gpu_step(w)
    want, _ = oracle_step(w)
    close(got, want, "prefill poison")


def test_prefill_with_one_query_equals_decode():
    w = workloads.make_custom(seq_lens=[5, 300, 129, 1000], num_q_heads=32, num_kv_heads=8,
                              head_dim=128, seed=92, q_lens=[1, 1, 1, 1])
    got, _ = gpu_step(w)
    want = oracle.decode_attention(w.q, *oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new,
                                                          w.block_table, w.seq_lens),
                                   w.block_table, w.seq_lens, w.scale)
    close(got, want, "prefill as decode")


def test_prefill_reruns_are_bit_identical():
    w = workloads.make_custom(seq_lens=[700, 1500], num_q_heads=16, num_kv_heads=4, head_dim=128,
                              seed=93, q_lens=[300, 77])
    _, dd = gpu_step(w)
    a = dd.prefill().clone()
    b = dd.prefill().clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_prefill_bad_page_and_short_seq_len_are_flagged():
    w = workloads.make_custom(seq_lens=[40, 40], num_q_heads=4, num_kv_heads=2, head_dim=64,
                              seed=94, q_lens=[10, 10])
    w.block_table[0, 1] = w.num_pages + 7
    dd = DeviceDecode(w)
    dd.make_prefill_plan()
    out = dd.prefill().float().cpu().numpy()
    assert dd.read_status() & binding.PA_DEV_BAD_PAGE
    assert np.all(np.isfinite(out))
    w2 = workloads.make_custom(seq_lens=[40, 40], num_q_heads=4, num_kv_heads=2, head_dim=64,
                               seed=95, q_lens=[10, 10])
    dd2 = DeviceDecode(w2)
    dd2.make_prefill_plan()
    dd2.seq_lens[1] = 5          # fewer cached tokens than the plan's queries
    dd2.prefill()
    assert dd2.read_status() & binding.PA_DEV_PLAN_MISMATCH


@pytest.mark.parametrize("cfg", [1, 2])
def test_prefill_benchmark_workload(cfg):
    """Both multi-token workloads at full size, every output (the oracle
    runs over a spawn-started process pool)."""
    w = workloads.make_prefill_config(cfg)
    got, _ = gpu_step(w)
    want = oracle_pool.prefill_all(("prefill_config", cfg))
    close(got, want, f"prefill workload {cfg}, all {got.shape[0] * got.shape[1]} rows x heads")


def test_prefill_whole_prompt():
    """q_lens = seq_lens: a whole 2048-token prompt attends causally over
    itself (512 tiles across the diagonal), every output against the oracle."""
    kw = dict(seq_lens=[2048, 300], num_q_heads=32, num_kv_heads=8, head_dim=128, seed=97,
              q_lens=[2048, 300])
    w = workloads.make_custom(**kw)
    got, _ = gpu_step(w)
    want = oracle_pool.prefill_all(("custom", kw))
    close(got, want, "whole prompt")


def test_prefill_benchmark_workload_mma_sync():
    """The piggybacked batch on the mma.sync kernel (64-row tiles), every output."""
    w = workloads.make_prefill_config(2)
    got, dd = gpu_step(w, rows_per_tile=64)
    assert dd.pf_plan.c.rows_per_tile == 64
    want = oracle_pool.prefill_all(("prefill_config", 2))
    close(got, want, "prefill workload 2 on mma.sync")


def _pools_match(dd, w):
    kp, vp = oracle.kv_append_tokens(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                     w.seq_lens, w.q_lens)
    ek = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    assert torch.equal(dd.k_pages, torch.from_numpy(kp).to(dd.k_pages.device).to(ek))
    assert torch.equal(dd.v_pages, torch.from_numpy(vp).to(dd.v_pages.device).to(ek))


def test_piggybacked_batch_on_two_streams():
    """The piggybacked workload served as an engine would: its single-token
    sequences through pa_append_decode_attention on a second stream, its
    prefill chunks through pa_kv_append_tokens + pa_prefill_attention.
    Every output row and every pool row match the oracle of the whole step."""
    w = workloads.make_prefill_config(2)
    assert np.sum(w.q_lens == 1) == 56
    dd = DeviceDecode(w)   # the pools
    ms = MixedStep(w)
    ms.run(dd.k_pages, dd.v_pages)
    assert ms.read_status() == 0
    got = ms.output().float().cpu().numpy()
    want = oracle_pool.prefill_all(("prefill_config", 2))
    close(got, want, "piggybacked batch on two streams, every output")
    _pools_match(dd, w)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("rows", [128, 64], ids=["tcgen05", "mma_sync"])
def test_mixed_batch_on_two_streams_small(dtype, rows):
    """Single-token and multi-token sequences interleaved in one batch (and a
    sequence with no query), on both multi-token kernels and element types."""
    w = workloads.make_custom(seq_lens=[700, 33, 260, 1, 1500, 96], q_lens=[1, 33, 1, 1, 200, 0],
                              num_q_heads=16, num_kv_heads=4, head_dim=128, seed=91, dtype=dtype)
    dd = DeviceDecode(w)
    ms = MixedStep(w, rows_per_tile=rows)
    ms.run(dd.k_pages, dd.v_pages)
    assert ms.read_status() == 0
    got = ms.output().float().cpu().numpy()
    want, _ = oracle_step(w)
    close(got, want, f"mixed batch on two streams, {dtype}, rows={rows}", dtype=dtype)
    _pools_match(dd, w)


@pytest.mark.parametrize("q_lens", [[1, 1, 1], [40, 7, 0]], ids=["decodes_only", "prefills_only"])
def test_mixed_batch_with_one_part_empty(q_lens):
    """A batch of only single-token sequences, or with none: the empty part
    makes no plan and launches nothing; the other part matches the oracle."""
    w = workloads.make_custom(seq_lens=[300, 45, 90], q_lens=q_lens, num_q_heads=8,
                              num_kv_heads=2, head_dim=128, seed=92)
    dd = DeviceDecode(w)
    ms = MixedStep(w)
    assert (ms.plan_d is None) == (len(ms.dec) == 0) and (ms.plan_p is None) == (len(ms.pre) == 0)
    ms.run(dd.k_pages, dd.v_pages)
    assert ms.read_status() == 0
    want, _ = oracle_step(w)
    close(ms.output().float().cpu().numpy(), want, f"mixed batch {q_lens}")
    _pools_match(dd, w)
