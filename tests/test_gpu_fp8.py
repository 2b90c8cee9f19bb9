"""GPU parity of the FP8 (E4M3) cache path (pa_kv_append_fp8,
pa_decode_attention_fp8, pa_append_decode_attention_fp8) against the float64
oracle, through the C ABI.

The append's codes and scales are compared bit for bit: both sides divide in
correctly rounded fp32 and round the quotient to the nearest E4M3 value,
ties to even.  Attention outputs use the fp16 path's tolerance.  Poisoned
workloads hold the E4M3 NaN pattern and NaN scales in every row no sequence
owns, so a read of one shows up in the output.
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


def oracle_fp8(w, heads=None):
    kc, vc, ks, vs = oracle.kv_append_fp8(w.k_codes, w.v_codes, w.k_scales, w.v_scales, w.k_new,
                                          w.v_new, w.block_table, w.seq_lens)
    out = oracle.decode_attention_fp8(w.q, kc, vc, ks, vs, w.block_table, w.seq_lens, w.scale,
                                      heads=heads)
    return out, (kc, vc, ks, vs)


def gpu_fp8(w, forced_splits=None, fused=False):
    dd = DeviceDecode(w)
    dd.make_plan(forced_splits=forced_splits)
    if fused:
        out = dd.append_decode_fp8()
    else:
        dd.append_fp8()
        out = dd.decode_fp8()
    status = dd.read_status()
    assert status == 0, f"device status {status:#x}"
    return out.cpu().numpy(), dd


def assert_pools_equal(dd, pools):
    kc, vc, ks, vs = pools
    assert np.array_equal(dd.k_codes.cpu().numpy(), kc)
    assert np.array_equal(dd.v_codes.cpu().numpy(), vc)
    assert np.array_equal(dd.k_scales.cpu().numpy().view(np.uint32), ks.view(np.uint32))
    assert np.array_equal(dd.v_scales.cpu().numpy().view(np.uint32), vs.view(np.uint32))


CASES = [
    # (seq_lens, Hq, Hkv, D, forced splits, dist)
    ([37, 100], 4, 2, 64, 1, ("uniform", 1.0)),
    ([1, 2, 15, 16, 17, 31, 33, 64], 8, 8, 128, 0, ("normal", 0.5)),     # G = 1
    ([5, 300, 129, 1000], 32, 8, 128, 0, ("normal", 0.5)),               # G = 4
    ([777, 50, 1], 16, 2, 128, 3, ("normal", 1.0)),                      # G = 8
    ([513, 257], 8, 1, 64, 5, ("uniform", 1.0)),                         # G = 8, D = 64
    ([2000, 3, 640], 4, 4, 64, 0, ("normal", 0.5)),                      # G = 1, D = 64
    ([96, 97, 1500], 16, 16, 128, 7, ("normal", 0.5)),
    ([250, 16], 32, 16, 64, 2, ("normal", 0.5)),                         # G = 2, D = 64
    ([300, 45, 1], 16, 8, 128, 0, ("normal", 0.5)),                      # G = 2
]


def _ids(c):
    return f"L{c[0][:3]}_G{c[1] // c[2]}_D{c[3]}_s{c[4]}"


def _make(case, salt, poison=False):
    lens, hq, hkv, d, splits, dist = case
    return workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                 dist=dist, seed=zlib.crc32(str(case).encode()) ^ salt,
                                 forced_splits=splits, poison=poison, kv="fp8")


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_fp8_parity_full(case):
    w = _make(case, 18)
    got, dd = gpu_fp8(w)
    want, pools = oracle_fp8(w)
    assert_close(got, want, f"fp8 {case}")
    assert_pools_equal(dd, pools)


@pytest.mark.parametrize("case", CASES + [([16, 32, 1, 17], 8, 2, 128, 0, ("normal", 0.5)),
                                          ([48, 9], 4, 4, 64, 3, ("uniform", 1.0))], ids=_ids)
def test_fp8_fused_append_decode_poisoned(case):
    """One launch gives the output and the pool bits of append then decode.
    Unowned rows hold NaN codes and NaN scales, the tail of each sequence's
    last page included: none of them may reach the output."""
    w = _make(case, 19, poison=True)
    got, dd = gpu_fp8(w, fused=True)
    want, pools = oracle_fp8(w)
    assert np.all(np.isfinite(got.astype(np.float32)))
    assert_close(got, want, f"fp8 fused {case}")
    assert_pools_equal(dd, pools)


def test_fp8_append_hand_worked_rows_bit_exact():
    """New rows built from the hand-worked E4M3 cases (ties to even,
    subnormals, an inexact scale, negative zero, an all-zero row): codes and
    scales match the oracle bit for bit."""
    D = 128
    rows = [[448, -1, 0.3125, 17, 19, -240, 0.005859375, 0.0048828125], [-224, 100, 3, 0.0625],
            [1.125, -0.5625, 0.001], [448, -0.0, 0, -0.0001], [0, 0, 0, 0]]
    w = workloads.make_custom(seq_lens=[3, 17, 40, 64, 1], num_q_heads=8, num_kv_heads=2,
                              head_dim=D, seed=51, kv="fp8")
    rng = np.random.default_rng(52)
    for b, r in enumerate(rows):
        for h in range(2):
            x = np.zeros(D, np.float16)
            x[rng.permutation(D)[:len(r)]] = np.array(r, np.float16)
            w.k_new[b, h] = x
            w.v_new[b, h] = -x
    dd = DeviceDecode(w)
    dd.append_fp8()
    assert dd.read_status() == 0
    _, pools = oracle_fp8(w, heads=[])
    assert_pools_equal(dd, pools)


def test_fp8_append_random_rows_bit_exact():
    """Rows of several magnitudes, every code and scale as the oracle's."""
    w = workloads.make_custom(seq_lens=list(range(1, 65)), num_q_heads=4, num_kv_heads=4,
                              head_dim=128, seed=53, kv="fp8")
    rng = np.random.default_rng(54)
    sd = np.exp2(rng.integers(-12, 6, size=(64, 4, 1)))
    w.k_new = (rng.standard_normal((64, 4, 128)) * sd).astype(np.float16)
    w.v_new = (rng.standard_normal((64, 4, 128)) * sd[::-1]).astype(np.float16)
    dd = DeviceDecode(w)
    dd.append_fp8()
    assert dd.read_status() == 0
    _, pools = oracle_fp8(w, heads=[])
    assert_pools_equal(dd, pools)


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_fp8_benchmark_config(cfg):
    w = workloads.make_config(cfg, kv="fp8")
    got, dd = gpu_fp8(w, fused=True)
    want, _ = oracle_fp8(w)
    assert_close(got, want, f"fp8 config {cfg}, every output")
    assert np.all(np.isfinite(got.astype(np.float32)))


def test_fp8_split_matches_unsplit():
    w = workloads.make_custom(seq_lens=[1500, 700, 33], num_q_heads=16, num_kv_heads=4,
                              head_dim=128, seed=55, kv="fp8")
    want, _ = oracle_fp8(w)
    for s in (1, 2, 5, 16, 0):
        got, _ = gpu_fp8(w, forced_splits=s)
        assert_close(got, want, f"fp8 splits={s}")


def test_fp8_zero_length_and_single_token():
    w = workloads.make_custom(seq_lens=[0, 1, 40, 0], num_q_heads=4, num_kv_heads=4, head_dim=64,
                              seed=56, kv="fp8")
    got, _ = gpu_fp8(w)
    want, _ = oracle_fp8(w)
    assert np.all(got[0] == 0) and np.all(got[3] == 0)
    assert_close(got, want, "zero and one token")


def test_fp8_bad_page_is_flagged_and_skipped():
    w = workloads.make_custom(seq_lens=[40, 40], num_q_heads=4, num_kv_heads=2, head_dim=64,
                              seed=57, kv="fp8")
    w.block_table[0, 1] = w.num_pages + 7
    dd = DeviceDecode(w)
    dd.make_plan()
    out = dd.decode_fp8().cpu().numpy()
    assert dd.read_status() & binding.PA_DEV_BAD_PAGE
    assert np.all(np.isfinite(out.astype(np.float32)))
    want1 = oracle.decode_attention_fp8(w.q, w.k_codes, w.v_codes, w.k_scales, w.v_scales,
                                        w.block_table, w.seq_lens, w.scale,
                                        heads=[(1, h) for h in range(4)])
    assert_close(out[1], want1[1], "sequence 1")


def test_fp8_and_int8_share_the_plan():
    """One plan and workspace serve the fp16, INT8 and FP8 calls of a shape."""
    lens = [300, 45, 1]
    wf = workloads.make_custom(seq_lens=lens, num_q_heads=16, num_kv_heads=8, head_dim=128,
                               seed=58, kv="fp8")
    wi = workloads.make_custom(seq_lens=lens, num_q_heads=16, num_kv_heads=8, head_dim=128,
                               seed=58, kv="int8")
    df, di = DeviceDecode(wf), DeviceDecode(wi)
    df.make_plan()
    di.plan_obj, di.workspace = df.plan_obj, df.workspace
    got_f = df.decode_fp8().cpu().numpy()
    got_i = di.decode_q8().cpu().numpy()
    assert df.read_status() == 0 and di.read_status() == 0
    assert_close(got_f, oracle.decode_attention_fp8(wf.q, wf.k_codes, wf.v_codes, wf.k_scales,
                                                    wf.v_scales, wf.block_table, wf.seq_lens,
                                                    wf.scale), "fp8")
    assert_close(got_i, oracle.decode_attention_q8(wi.q, wi.k_codes, wi.v_codes, wi.k_scales,
                                                   wi.v_scales, wi.block_table, wi.seq_lens,
                                                   wi.scale), "int8")


@pytest.mark.parametrize("case", [c for c in CASES if c[3] == 128], ids=_ids)
def test_fp8_both_page_stage_counts(case):
    """Plans forced to 2 and to 3 page stages per warp give the oracle's
    outputs and the same pools."""
    lens, hq, hkv, d, splits, dist = case
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              dist=dist, seed=zlib.crc32(str(case).encode()) ^ 28,
                              forced_splits=splits, kv="fp8")
    want, pools = oracle_fp8(w)
    for ns in (2, 3):
        dd = DeviceDecode(w)
        dd.make_plan(q8_stages=ns)
        assert dd.plan_obj.c.q8_stages == ns
        got = dd.append_decode_fp8().cpu().numpy()
        assert dd.read_status() == 0
        assert_close(got, want, f"fp8 {case} stages={ns}")
        assert_pools_equal(dd, pools)
