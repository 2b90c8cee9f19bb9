"""GPU parity: the CUDA path against the float64 oracle, through the C ABI.

Small and medium cases are compared on every output.  They cover several
pages, ragged tails, every G and D built, and forced and automatic splits.
The five benchmark workloads run at full size, in the launch configuration
the benchmark times, and are compared on sampled (sequence, head) outputs.
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


def run_step(w, forced_splits=None):
    """append + plan + decode on the GPU; returns (out fp16 numpy, DeviceDecode)."""
    dd = DeviceDecode(w)
    dd.append()
    dd.make_plan(forced_splits=forced_splits)
    out = dd.decode()
    status = dd.read_status()
    assert status == 0, f"device status {status:#x}"
    return out.cpu().numpy(), dd


def oracle_step(w, heads=None):
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    return oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale, heads=heads)


# ---------------------------------------------------------------------------
# full comparison on small/medium shapes

CASES = [
    # (seq_lens, Hq, Hkv, D, forced splits, dist)
    ([37, 100], 4, 2, 64, 1, ("uniform", 1.0)),
    ([1, 2, 15, 16, 17, 31, 33, 64], 8, 8, 128, 0, ("normal", 0.5)),
    ([5, 300, 129, 1000], 32, 8, 128, 0, ("normal", 0.5)),
    ([777, 50, 1], 16, 2, 128, 3, ("normal", 1.0)),
    ([513, 257], 8, 1, 64, 5, ("uniform", 1.0)),
    ([2000, 3, 640], 4, 4, 64, 0, ("normal", 0.5)),
    ([96, 97, 1500], 16, 16, 128, 7, ("normal", 0.5)),
    ([300, 45], 16, 2, 128, 0, ("normal", 0.5)),     # G = 8
    ([250, 16], 32, 4, 64, 2, ("normal", 0.5)),      # G = 8, D = 64
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"L{c[0][:3]}_G{c[1]//c[2]}_D{c[3]}_s{c[4]}")
def test_parity_full(case):
    lens, hq, hkv, d, splits, dist = case
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              dist=dist, seed=zlib.crc32(str(case).encode()), forced_splits=splits)
    got, _ = run_step(w)
    assert_close(got, oracle_step(w), str(case))


def test_parity_config1_full():
    w = workloads.make_config(1)
    got, dd = run_step(w)
    assert_close(got, oracle_step(w), "config 1")
    assert dd.plan_obj.c.num_groups == 0


def test_poisoned_pool_never_read():
    """Unowned rows hold NaN: any read past a sequence's end would show."""
    w = workloads.make_custom(seq_lens=[1, 17, 250, 33], num_q_heads=8, num_kv_heads=2,
                              head_dim=128, seed=21, poison=True)
    for splits in (0, 1, 4):
        got, _ = run_step(w, forced_splits=splits)
        assert_close(got, oracle_step(w), f"poison splits={splits}")


# ---------------------------------------------------------------------------
# full-size benchmark workloads, every output against the oracle

@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_parity_benchmark_config(cfg):
    w = workloads.make_config(cfg)
    got, dd = run_step(w)
    want = oracle_step(w)
    assert_close(got, want, f"config {cfg}, all {w.batch * w.num_q_heads} heads")
    assert np.all(np.isfinite(got.astype(np.float32)))
    if cfg == 2:
        assert dd.plan_obj.c.max_splits == 16


# ---------------------------------------------------------------------------
# fused append + decode: same output as append then decode, same pool bits

FUSED = CASES + [
    ([16, 32, 1, 17], 8, 2, 128, 0, ("normal", 0.5)),    # new token in row 15 / row 0
    ([48, 9], 4, 4, 64, 3, ("uniform", 1.0)),
]


@pytest.mark.parametrize("case", FUSED, ids=lambda c: f"L{c[0][:3]}_G{c[1]//c[2]}_D{c[3]}_s{c[4]}")
def test_fused_append_decode(case):
    lens, hq, hkv, d, splits, dist = case
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              dist=dist, seed=zlib.crc32(str(case).encode()) ^ 7,
                              forced_splits=splits, poison=True)
    dd = DeviceDecode(w)
    dd.make_plan()
    got = dd.append_decode().cpu().numpy()
    assert dd.read_status() == 0
    assert_close(got, oracle_step(w), f"fused {case}")
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    assert np.array_equal(dd.k_pages.cpu().numpy().view(np.uint16), kp.view(np.uint16))
    assert np.array_equal(dd.v_pages.cpu().numpy().view(np.uint16), vp.view(np.uint16))


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_fused_append_decode_benchmark_config(cfg):
    """The bench's launch: the fused call with the automatic plan (workload 2
    forces its 16 splits), every output against the oracle."""
    w = workloads.make_config(cfg)
    dd = DeviceDecode(w)
    dd.make_plan()
    got = dd.append_decode().cpu().numpy()
    assert dd.read_status() == 0
    want = oracle_step(w)
    assert_close(got, want, f"fused config {cfg}")
    # the new rows landed in the pool
    slots = oracle.gather_slots(w.block_table, w.seq_lens, 16)
    kp = dd.k_pages.cpu().numpy()
    for b in range(w.batch):
        s = int(slots[b, int(w.seq_lens[b]) - 1])
        assert np.array_equal(kp[s // 16, :, s % 16].view(np.uint16), w.k_new[b].view(np.uint16))


# ---------------------------------------------------------------------------
# exact index and byte checks

@pytest.mark.parametrize("cfg", [1, 5])
def test_gather_indices_exact(cfg):
    w = workloads.make_config(cfg)
    dd = DeviceDecode(w)
    slots = dd.gather_slots().cpu().numpy()
    assert dd.read_status() == 0
    assert np.array_equal(slots.astype(np.int64), oracle.gather_slots(w.block_table, w.seq_lens, 16))


def test_gather_indices_ragged():
    w = workloads.make_custom(seq_lens=[0, 1, 16, 17, 95], num_q_heads=2, num_kv_heads=1,
                              head_dim=64, seed=22, max_pages_per_seq=9)
    dd = DeviceDecode(w)
    slots = dd.gather_slots().cpu().numpy()
    assert np.array_equal(slots.astype(np.int64), oracle.gather_slots(w.block_table, w.seq_lens, 16))


@pytest.mark.parametrize("cfg", [1, 3])
def test_append_bit_exact(cfg):
    w = workloads.make_config(cfg)
    dd = DeviceDecode(w)
    dd.append()
    assert dd.read_status() == 0
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    assert np.array_equal(dd.k_pages.cpu().numpy().view(np.uint16), kp.view(np.uint16))
    assert np.array_equal(dd.v_pages.cpu().numpy().view(np.uint16), vp.view(np.uint16))


# ---------------------------------------------------------------------------
# invariants

def test_page_permutation_bit_identical():
    w = workloads.make_custom(seq_lens=[37, 400, 5, 129], num_q_heads=8, num_kv_heads=2,
                              head_dim=128, seed=23)
    ref, _ = run_step(w)
    perm = np.random.default_rng(24).permutation(w.num_pages)
    w2 = workloads.make_custom(seq_lens=[37, 400, 5, 129], num_q_heads=8, num_kv_heads=2,
                               head_dim=128, seed=23)
    w2.k_pages = np.empty_like(w.k_pages)
    w2.v_pages = np.empty_like(w.v_pages)
    w2.k_pages[perm] = w.k_pages
    w2.v_pages[perm] = w.v_pages
    w2.block_table = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    got, _ = run_step(w2)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_split_matches_unsplit():
    w = workloads.make_custom(seq_lens=[1500, 700, 33], num_q_heads=16, num_kv_heads=4,
                              head_dim=128, seed=25)
    base, _ = run_step(w, forced_splits=1)
    want = oracle_step(w)
    for s in (2, 5, 16, 0):
        got, _ = run_step(w, forced_splits=s)
        assert_close(got, want, f"splits={s}")
        assert_close(got, base.astype(np.float64), f"splits={s} vs unsplit")


def test_seq_len_one_returns_v_exactly():
    w = workloads.make_custom(seq_lens=[1, 1, 1], num_q_heads=8, num_kv_heads=2, head_dim=128, seed=26)
    got, _ = run_step(w)
    for b in range(3):
        for h in range(8):
            assert np.array_equal(got[b, h].view(np.uint16), w.v_new[b, h // 4].view(np.uint16))


def test_zero_length_sequences_give_zeros():
    w = workloads.make_custom(seq_lens=[0, 40, 0], num_q_heads=4, num_kv_heads=4, head_dim=64, seed=27)
    got, _ = run_step(w)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert_close(got[1], oracle_step(w)[1], "middle sequence")


def test_rerun_is_bit_identical():
    w = workloads.make_config(5)
    dd = DeviceDecode(w)
    dd.append()
    dd.make_plan()
    a = dd.decode().clone()
    b = dd.decode().clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------------------
# device-detected problems are flagged, never trapped

def test_bad_page_index_is_flagged_and_skipped():
    w = workloads.make_custom(seq_lens=[40, 40], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=28)
    want = oracle_step(w)
    w.block_table[0, 1] = w.num_pages + 7   # sequence 0, page 1: out of range
    dd = DeviceDecode(w)
    dd.make_plan()
    out = dd.decode().cpu().numpy()
    assert dd.read_status() & binding.PA_DEV_BAD_PAGE
    assert np.all(np.isfinite(out.astype(np.float32)))
    # sequence 1 is untouched by the bad entry
    kp, vp = w.k_pages, w.v_pages
    want1 = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale, heads=[(1, h) for h in range(4)])
    assert_close(out[1], want1[1], "sequence 1")
    del want


def test_negative_page_index_in_append_is_flagged():
    w = workloads.make_custom(seq_lens=[20], num_q_heads=2, num_kv_heads=2, head_dim=64, seed=29)
    w.block_table[0, 1] = -3
    dd = DeviceDecode(w)
    before = dd.k_pages.clone()
    dd.append()
    assert dd.read_status() & binding.PA_DEV_BAD_PAGE
    assert torch.equal(before, dd.k_pages)


def test_workspace_without_plan_is_flagged():
    w = workloads.make_custom(seq_lens=[50, 20], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=30)
    dd = DeviceDecode(w)
    plan = binding.Plan(dd.shape, w.seq_lens, dd.num_sms, 0)
    plan_b = binding.Plan(dd.shape, w.seq_lens, dd.num_sms, 3)
    assert plan_b.structure() != plan.structure()
    ws = torch.zeros(max(plan.workspace_bytes, plan_b.workspace_bytes), dtype=torch.uint8,
                     device="cuda")   # never uploaded
    dd.out.fill_(0)
    binding.decode(dd.shape, plan, dd.q, dd.k_pages, dd.v_pages, dd.block_table, dd.seq_lens,
                   w.scale, dd.out, ws, dd.status)
    assert dd.read_status() & binding.PA_DEV_PLAN_MISMATCH
    # a stale plan: upload plan A, decode with plan B whose task list differs
    binding.upload(plan, ws)
    dd.status.zero_()
    binding.decode(dd.shape, plan_b, dd.q, dd.k_pages, dd.v_pages, dd.block_table, dd.seq_lens,
                   w.scale, dd.out, ws, dd.status)
    assert dd.read_status() & binding.PA_DEV_PLAN_MISMATCH


def test_device_seq_lens_longer_than_plan_are_flagged():
    w = workloads.make_custom(seq_lens=[150, 60], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=31)
    dd = DeviceDecode(w)
    dd.make_plan(seq_lens_host=np.array([100, 60], np.int32))
    dd.decode()
    assert dd.read_status() & binding.PA_DEV_PLAN_MISMATCH


def test_device_seq_len_out_of_range_is_flagged():
    w = workloads.make_custom(seq_lens=[30, 30], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=32)
    dd = DeviceDecode(w)
    dd.make_plan()
    dd.seq_lens[0] = w.max_pages_per_seq * 16 + 100
    dd.decode()
    assert dd.read_status() & binding.PA_DEV_BAD_SEQ_LEN


def test_maximum_split_count():
    """A request for more splits than the limit is clamped to 1024 page-aligned
    splits (two pages each here). The split merge then combines 1024 partials
    per head, and the result still matches the unsplit oracle."""
    w = workloads.make_custom(seq_lens=[32768, 40], num_q_heads=8, num_kv_heads=2, head_dim=64,
                              seed=29)
    dd = DeviceDecode(w)
    dd.append()
    dd.make_plan(forced_splits=5000)
    assert int(dd.plan_obj.c.max_splits) == 1024
    got = dd.decode().cpu().numpy()
    assert dd.read_status() == 0
    assert_close(got, oracle_step(w), "1024 splits")
