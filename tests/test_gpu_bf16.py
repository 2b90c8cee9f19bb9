"""GPU parity of the bf16 path (pa_shape_t.dtype = PA_DTYPE_BF16: q, K, V,
new rows and out in bf16) against the float64 oracle, through the C ABI.

Inputs are bf16 numbers held as float32 on the host, so the oracle widens
them exactly.  The append is a bit copy and is compared bit for bit; the
outputs use the bf16 tolerance of tests/parity.py.
"""

from __future__ import annotations

import zlib

import numpy as np
import pytest

import oracle
from paged_kv_decode_24_gb300 import binding, workloads
from paged_kv_decode_24_gb300.runner import DeviceDecode
from tests.parity import assert_close
from tests.test_gpu_parity import CASES

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


def oracle_step(w, heads=None):
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    return oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale, heads=heads)


def gpu_step(w, forced_splits=None, fused=False):
    dd = DeviceDecode(w)
    assert dd.q.dtype == torch.bfloat16 and dd.shape.dtype == binding.PA_DTYPE_BF16
    dd.make_plan(forced_splits=forced_splits)
    if fused:
        out = dd.append_decode()
    else:
        dd.append()
        out = dd.decode()
    status = dd.read_status()
    assert status == 0, f"device status {status:#x}"
    return out.float().cpu().numpy(), dd


def bf16_bits(a_f32):
    """Bits of bf16-exact float32 values as bf16 (the top half of each word)."""
    return (np.ascontiguousarray(a_f32, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _ids(c):
    return f"L{c[0][:3]}_G{c[1] // c[2]}_D{c[3]}_s{c[4]}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_bf16_parity_full(case):
    lens, hq, hkv, d, splits, dist = case
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              dist=dist, seed=zlib.crc32(str(case).encode()) ^ 16,
                              forced_splits=splits, dtype="bf16")
    got, dd = gpu_step(w)
    assert_close(got, oracle_step(w), f"bf16 {case}", dtype="bf16")
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    assert np.array_equal(dd.k_pages.view(torch.int16).cpu().numpy().view(np.uint16), bf16_bits(kp))
    assert np.array_equal(dd.v_pages.view(torch.int16).cpu().numpy().view(np.uint16), bf16_bits(vp))


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_bf16_fused_append_decode(case):
    """Unowned rows hold NaN: a read past a sequence's end would show."""
    lens, hq, hkv, d, splits, dist = case
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              dist=dist, seed=zlib.crc32(str(case).encode()) ^ 17,
                              forced_splits=splits, poison=True, dtype="bf16")
    got, dd = gpu_step(w, fused=True)
    assert_close(got, oracle_step(w), f"bf16 fused {case}", dtype="bf16")
    kp, _ = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    # unowned rows are NaN, whose bf16 bit pattern depends on the converter
    assert np.array_equal(dd.k_pages.float().cpu().numpy(), kp, equal_nan=True)


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_bf16_benchmark_config(cfg):
    w = workloads.make_config(cfg, dtype="bf16")
    got, dd = gpu_step(w, fused=True)
    want = oracle_step(w)
    assert_close(got, want, f"bf16 config {cfg}, every output", dtype="bf16")


def test_bf16_seq_len_one_returns_v_exactly():
    w = workloads.make_custom(seq_lens=[1, 1, 1], num_q_heads=8, num_kv_heads=2, head_dim=128,
                              seed=51, dtype="bf16")
    got, _ = gpu_step(w)
    for b in range(3):
        for h in range(8):
            assert np.array_equal(got[b, h].astype(np.float32), w.v_new[b, h // 4])
    w1 = workloads.make_custom(seq_lens=[1, 1], num_q_heads=4, num_kv_heads=4, head_dim=64,
                               seed=52, dtype="bf16")
    got1, _ = gpu_step(w1)
    assert np.array_equal(got1.astype(np.float32), w1.v_new)


def test_bf16_split_matches_unsplit_and_reruns_are_identical():
    w = workloads.make_custom(seq_lens=[1500, 700, 33], num_q_heads=16, num_kv_heads=4,
                              head_dim=128, seed=53, dtype="bf16")
    want = oracle_step(w)
    for s in (1, 2, 5, 0):
        got, dd = gpu_step(w, forced_splits=s)
        assert_close(got, want, f"bf16 splits={s}", dtype="bf16")
    a = dd.decode().clone()
    b = dd.decode().clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bf16_static_workspace_entry():
    w = workloads.make_custom(seq_lens=[300, 45, 1], num_q_heads=16, num_kv_heads=8, head_dim=128,
                              seed=54, dtype="bf16")
    dd = DeviceDecode(w)
    dd.append()
    plan = binding.Plan(dd.shape, w.seq_lens, dd.num_sms, 3)
    out = torch.empty_like(dd.q)
    binding.decode_static(dd.shape, plan, dd.q, dd.k_pages, dd.v_pages, dd.block_table,
                          dd.seq_lens, w.scale, out, dd.status)
    assert dd.read_status() == 0
    assert_close(out.float().cpu().numpy(), oracle_step(w), "bf16 static", dtype="bf16")
