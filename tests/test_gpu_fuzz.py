"""GPU parity over seeded random configurations, against the float64 oracle.

Each case draws a shape and a launch setting at random: the cache (fp16,
bf16, INT8, FP8), the group size and head dimension, ragged sequence lengths
(zero, one page, page boundaries, thousands of tokens), the split policy
(automatic, or forced), the merge form, the SM count the plan is made for
(small counts make the planner bundle short tasks one per warp), the 8-bit
kernel's page stages, the fused or separate append, and (fused) the early
page copies of plan option early_kv.  The multi-token cases draw query
counts per sequence and both tile kernels, and the mixed cases serve
batches of single-token and multi-token sequences on two streams.  Every output is compared at the path's tolerance, and the
appended pools bit for bit.
"""

from __future__ import annotations

import numpy as np
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


def _lengths(rng, n):
    pick = rng.choice(["zero", "one", "edge", "short", "long"], size=n,
                      p=[0.05, 0.1, 0.25, 0.35, 0.25])
    out = []
    for k in pick:
        if k == "zero":
            out.append(0)
        elif k == "one":
            out.append(1)
        elif k == "edge":
            out.append(int(16 * rng.integers(1, 40) + rng.choice([-1, 0, 1])))
        elif k == "short":
            out.append(int(rng.integers(2, 300)))
        else:
            out.append(int(rng.integers(300, 3000)))
    return [max(0, x) for x in out]


def _decode_case(seed):
    rng = np.random.default_rng(seed)
    kv = str(rng.choice(["fp16", "bf16", "int8", "fp8"]))
    d = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4, 8]))
    hkv = int(rng.choice([1, 2, 4]))
    lens = _lengths(rng, int(rng.integers(1, 12)))
    if max(lens) == 0:
        lens[0] = 17
    return dict(kv=kv, d=d, g=g, hkv=hkv, lens=lens,
                splits=int(rng.choice([0, 0, 1, 2, 3, 7, 16])),
                merge=str(rng.choice(["split", "combine"])),
                sms=int(rng.choice([1, 2, 8, 152])),
                stages=int(rng.choice([0, 2, 3])),
                fused=bool(rng.integers(0, 2)),
                dist=("normal", float(rng.choice([0.5, 1.0]))),
                early=bool(rng.integers(0, 2)))


DECODE_SEEDS = list(range(7100, 7260))


@pytest.mark.parametrize("seed", DECODE_SEEDS)
def test_random_decode_case(seed):
    c = _decode_case(seed)
    dtype = "bf16" if c["kv"] == "bf16" else "fp16"
    cache = c["kv"] if c["kv"] in ("int8", "fp8") else "fp16"
    w = workloads.make_custom(seq_lens=c["lens"], num_q_heads=c["hkv"] * c["g"],
                              num_kv_heads=c["hkv"], head_dim=c["d"], dist=c["dist"], seed=seed,
                              forced_splits=c["splits"], kv=cache, dtype=dtype,
                              poison=cache == "fp8")
    dd = DeviceDecode(w, num_sms=c["sms"])
    opts = dict(merge=c["merge"])
    if c["stages"]:
        opts["q8_stages"] = c["stages"]
    if c["fused"] and c["early"]:   # (after a separate append kernel it would not hold)
        opts["early_kv"] = 1
    dd.make_plan(**opts)
    if cache == "fp16":
        if c["fused"]:
            got = dd.append_decode()
        else:
            dd.append()
            got = dd.decode()
        kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                  w.seq_lens)
        want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
        pools = [(dd.k_pages, kp), (dd.v_pages, vp)]
    else:
        if c["fused"]:
            got = dd.append_decode8()
        else:
            dd.append8()
            got = dd.decode8()
        want, (kc, vc, ks, vs) = oracle_append_decode(w)
        pools = [(dd.k_codes, kc), (dd.v_codes, vc), (dd.k_scales, ks), (dd.v_scales, vs)]
    status = dd.read_status()
    assert status == 0, (c, f"{status:#x}")
    assert_close(got.float().cpu().numpy(), want, f"random decode case {seed}: {c}", dtype=dtype)
    _pools_bit_exact(pools, c)


def _pools_bit_exact(pools, c):
    """Device pools against the oracle's, byte for byte (NaN patterns too)."""
    for dev, host in pools:
        got = dev.cpu()
        want = torch.from_numpy(np.ascontiguousarray(host)).to(got.dtype)
        assert torch.equal(got.view(torch.uint8), want.view(torch.uint8)), c


def _prefill_case(seed):
    rng = np.random.default_rng(seed)
    lens = [max(1, x) for x in _lengths(rng, int(rng.integers(1, 7)))]
    qls = [int(rng.integers(0, L + 1)) if rng.random() < 0.7 else int(min(L, 1)) for L in lens]
    return dict(lens=lens, qls=qls, d=int(rng.choice([64, 128])), g=int(rng.choice([1, 2, 4, 8])),
                hkv=int(rng.choice([1, 2, 4])), rows=int(rng.choice([128, 64])),
                dtype=str(rng.choice(["fp16", "bf16"])))


PREFILL_SEEDS = list(range(7300, 7348))


@pytest.mark.parametrize("seed", PREFILL_SEEDS)
def test_random_multi_token_case(seed):
    c = _prefill_case(seed)
    w = workloads.make_custom(seq_lens=c["lens"], q_lens=c["qls"],
                              num_q_heads=c["hkv"] * c["g"], num_kv_heads=c["hkv"],
                              head_dim=c["d"], seed=seed, dtype=c["dtype"])
    dd = DeviceDecode(w)
    dd.make_prefill_plan(rows_per_tile=c["rows"])
    dd.append_tokens()
    got = dd.prefill()
    status = dd.read_status()
    assert status == 0, (c, f"{status:#x}")
    kp, vp = oracle.kv_append_tokens(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                     w.seq_lens, w.q_lens)
    want = oracle.prefill_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.q_lens, w.scale)
    assert_close(got.float().cpu().numpy(), want, f"random multi-token case {seed}: {c}",
                 dtype=c["dtype"])
    _pools_bit_exact([(dd.k_pages, kp), (dd.v_pages, vp)], c)


MIXED_SEEDS = list(range(7400, 7412))


@pytest.mark.parametrize("seed", MIXED_SEEDS)
def test_random_mixed_batch_on_two_streams(seed):
    """Random batches of single-token and multi-token sequences served by
    MixedStep (decode call on a second stream beside the multi-token call)."""
    from paged_kv_decode_24_gb300.runner import MixedStep
    rng = np.random.default_rng(seed)
    lens = [max(1, x) for x in _lengths(rng, int(rng.integers(2, 9)))]
    qls = [1 if rng.random() < 0.5 else int(rng.integers(0, L + 1)) for L in lens]
    g, hkv = int(rng.choice([1, 2, 4, 8])), int(rng.choice([1, 2, 4]))
    dtype = str(rng.choice(["fp16", "bf16"]))
    w = workloads.make_custom(seq_lens=lens, q_lens=qls, num_q_heads=hkv * g, num_kv_heads=hkv,
                              head_dim=int(rng.choice([64, 128])), seed=seed, dtype=dtype)
    dd = DeviceDecode(w)
    ms = MixedStep(w, rows_per_tile=int(rng.choice([128, 64])),
                   decode_sms=int(rng.choice([1, 16, 50])))
    ms.run(dd.k_pages, dd.v_pages)
    assert ms.read_status() == 0, (lens, qls)
    kp, vp = oracle.kv_append_tokens(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                     w.seq_lens, w.q_lens)
    want = oracle.prefill_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.q_lens, w.scale)
    assert_close(ms.output().float().cpu().numpy(), want, f"random mixed batch {seed}",
                 dtype=dtype)
    _pools_bit_exact([(dd.k_pages, kp), (dd.v_pages, vp)], (lens, qls))
