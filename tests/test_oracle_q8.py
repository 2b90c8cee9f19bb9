"""Pins of the INT8-cache oracle (oracle/quant.py) against what the
quantisation rule and mathematics fix.  No GPU.

* Rows worked by hand (tests/golden/int8_rows.txt): exact scales and codes,
  ties to even, and attention over dequantised rows with per-row scales.
* The rounding bound: every code is within half a step of x / scale, and the
  largest magnitude of a nonzero row maps to +-127.
* A reduction to the fp16 oracle: when every code * scale is exact in fp16,
  attention over the INT8 cache equals attention over that fp16 cache.
* Append: only the new slot changes, and it holds the new row's codes.
A copy of the oracle with a planted mistake must fail at least one pin.
"""

from __future__ import annotations

import math
import os
import types

import numpy as np
import pytest

import oracle
from oracle import quant as oracle_quant
from paged_kv_decode_24_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int8_rows.txt")


def _parse():
    rows, attends, cur = [], [], None
    with open(GOLDEN) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("row ") or line.startswith("attend "):
                kind, name = line.split(None, 1)
                cur = {"name": name}
                (rows if kind == "row" else attends).append(cur)
                continue
            key, val = (x.strip() for x in line.split("=", 1))
            if key == "scale" and "math" in val:
                cur[key] = float(eval(val, {"math": math}))
            elif ";" in val or key in ("k_codes", "v_codes"):
                cur[key] = np.array([[float(x) for x in r.split()] for r in val.split(";")])
            else:
                cur[key] = np.array([float(x) for x in val.split()])
    return rows, attends


ROWS, ATTENDS = _parse()


# --------------------------------------------------------------------------
# checks, written against an oracle module so planted mistakes can be tried

def check_golden_rows(orc):
    bad = 0
    for r in ROWS:
        x = r["x"].astype(np.float16)
        codes, scale = orc.quantize_rows_int8(x[None, :])
        bad += int(float(scale[0]) != float(r["scale"][0]))
        bad += int(not np.array_equal(codes[0].astype(np.int64), r["codes"].astype(np.int64)))
    return bad


def check_golden_attend(orc):
    worst = 0.0
    S = 2
    for c in ATTENDS:
        L, D = c["k_codes"].shape
        pages = [int(p) for p in np.atleast_1d(c["pages"])]
        P = max(pages) + 1
        kc = np.full((P, 1, S, D), 99, np.int8)        # junk outside the sequence
        vc = np.full((P, 1, S, D), -99, np.int8)
        ks = np.full((P, 1, S), 7.0, np.float32)
        vs = np.full((P, 1, S), 7.0, np.float32)
        for t in range(L):
            kc[pages[t // S], 0, t % S] = c["k_codes"][t]
            vc[pages[t // S], 0, t % S] = c["v_codes"][t]
            ks[pages[t // S], 0, t % S] = c["k_scales"][t]
            vs[pages[t // S], 0, t % S] = c["v_scales"][t]
        bt = np.array([pages], np.int32)
        got = orc.decode_attention_q8(c["q"][None, None, :], kc, vc, ks, vs, bt, np.array([L]),
                                      c["scale"])
        worst = max(worst, float(np.max(np.abs(got[0, 0] - c["expect"]))))
    return worst


def check_rounding_bound(orc, seed=31):
    """Worst violation of |x/scale - code| <= 1/2 (+ fp32 slack), of
    max|code| = 127 on nonzero rows, and of scale = nearest fp32 to amax/127."""
    rng = np.random.default_rng(seed)
    bad = 0
    for sd in (1e-4, 0.02, 0.5, 3.0, 200.0):
        x = (rng.standard_normal((64, 128)) * sd).astype(np.float16)
        codes, scales = orc.quantize_rows_int8(x)
        xf = x.astype(np.float64)
        amax = np.abs(xf).max(axis=1)
        s64 = scales.astype(np.float64)
        ulp = np.spacing(scales).astype(np.float64)
        bad += int(np.sum(np.abs(s64 - amax / 127.0) > ulp / 2))
        ratio = xf / s64[:, None]
        bad += int(np.sum(np.abs(ratio - codes) > 0.5 + 1e-5))
        bad += int(np.sum(np.abs(codes.astype(np.int64)).max(axis=1) != 127))
    return bad


def check_exact_reduces_to_fp16(orc, seed=32):
    """Codes times power-of-two scales are exact in fp16: the INT8 oracle must
    equal the fp16 oracle on that fp16 cache, bit for bit."""
    rng = np.random.default_rng(seed)
    w = workloads.make_custom(seq_lens=[1, 19, 40, 16], num_q_heads=8, num_kv_heads=2,
                              head_dim=16, seed=33)
    shape = w.k_pages.shape
    kc = rng.integers(-127, 128, size=shape).astype(np.int8)
    vc = rng.integers(-127, 128, size=shape).astype(np.int8)
    ks = np.ldexp(1.0, rng.integers(-10, 1, size=shape[:3])).astype(np.float32)
    vs = np.ldexp(1.0, rng.integers(-10, 1, size=shape[:3])).astype(np.float32)
    kp = (kc.astype(np.float64) * ks[..., None]).astype(np.float16)
    vp = (vc.astype(np.float64) * vs[..., None]).astype(np.float16)
    ref = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
    got = orc.decode_attention_q8(w.q, kc, vc, ks, vs, w.block_table, w.seq_lens, w.scale)
    return float(np.max(np.abs(got - ref)))


def check_append(orc, seed=34):
    """Only the new slots change; they hold the new rows' codes within half a
    step; every other byte of the pools is untouched."""
    w = workloads.make_custom(seq_lens=[1, 16, 17, 40], num_q_heads=2, num_kv_heads=2,
                              head_dim=8, seed=seed)
    rng = np.random.default_rng(seed)
    shape = w.k_pages.shape
    kc = rng.integers(-127, 128, size=shape).astype(np.int8)
    vc = rng.integers(-127, 128, size=shape).astype(np.int8)
    ks = rng.random(shape[:3]).astype(np.float32)
    vs = rng.random(shape[:3]).astype(np.float32)
    kc2, vc2, ks2, vs2 = orc.kv_append_q8(kc, vc, ks, vs, w.k_new, w.v_new, w.block_table,
                                          w.seq_lens)
    S = 16
    bad = 0
    touched = set()
    for b, L in enumerate(w.seq_lens):
        page, slot = int(w.block_table[b, (L - 1) // S]), (L - 1) % S
        touched.add((page, slot))
        for new, c2, s2 in ((w.k_new[b], kc2, ks2), (w.v_new[b], vc2, vs2)):
            deq = c2[page, :, slot].astype(np.float64) * s2[page, :, slot, None].astype(np.float64)
            step = s2[page, :, slot, None].astype(np.float64)
            bad += int(np.sum(np.abs(deq - new.astype(np.float64)) > 0.5 * step * (1 + 1e-5)))
    for (a, a2) in ((kc, kc2), (vc, vc2), (ks, ks2), (vs, vs2)):
        diff = np.argwhere(np.any((a != a2).reshape(shape[0], shape[1], S, -1), axis=(1, 3)))
        bad += len(set((int(p), int(s)) for p, s in diff) - touched)
    return bad


# --------------------------------------------------------------------------
# the pins

def test_golden_rows():
    assert check_golden_rows(oracle) == 0


def test_golden_attend_over_dequantised_rows():
    assert check_golden_attend(oracle) < 1e-12


def test_rounding_bound_and_full_range():
    assert check_rounding_bound(oracle) == 0


def test_exact_codes_reduce_to_fp16_oracle():
    assert check_exact_reduces_to_fp16(oracle) == 0.0


def test_append_writes_only_the_new_slot():
    assert check_append(oracle) == 0


def test_zero_row_and_seq_len_zero():
    codes, scales = oracle.quantize_rows_int8(np.zeros((3, 16), np.float16))
    assert np.all(codes == 0) and np.all(scales == 0)
    w = workloads.make_custom(seq_lens=[0, 3], num_q_heads=2, num_kv_heads=1, head_dim=8, seed=35)
    shape = w.k_pages.shape
    kc = np.ones(shape, np.int8)
    ks = np.ones(shape[:3], np.float32)
    got = oracle.decode_attention_q8(w.q, kc, kc, ks, ks, w.block_table, w.seq_lens, w.scale)
    assert np.all(got[0] == 0.0)
    np.testing.assert_allclose(got[1], 1.0, rtol=0, atol=1e-15)   # every V row is all ones


# --------------------------------------------------------------------------
# planted mistakes

def _mutant(**overrides):
    m = types.ModuleType("oracle_quant_mutant")
    m.__dict__.update(vars(oracle_quant))
    m.__dict__.update(overrides)
    for name, fn in list(m.__dict__.items()):
        if isinstance(fn, types.FunctionType) and name not in overrides:
            m.__dict__[name] = types.FunctionType(fn.__code__, m.__dict__, name, fn.__defaults__)
    return m


def _mutants():
    def truncating(x):
        x32 = np.asarray(x).astype(np.float32)
        s = (np.max(np.abs(x32), axis=-1) / np.float32(127)).astype(np.float32)
        safe = np.where(s > 0, s, np.float32(1))
        return np.trunc(x32 / safe[..., None]).astype(np.int8), s

    def scale_of_slot_zero(codes, scales, block_table, b, seq_len, kv_head):
        S = codes.shape[2]
        t = np.arange(seq_len)
        phys = block_table[b, t // S].astype(np.int64)
        return codes[phys, kv_head, t % S, :].astype(np.float64) * \
            scales[phys, kv_head, 0].astype(np.float64)[:, None]

    def no_scale(codes, scales):
        return codes.astype(np.float64)

    def swapped_kv_scales(q, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens, scale,
                          heads=None):
        return oracle_quant.decode_attention_q8(q, k_codes, v_codes, v_scales, k_scales,
                                                block_table, seq_lens, scale, heads)

    def append_to_next_slot(k_codes, v_codes, k_scales, v_scales, k_new, v_new, block_table,
                            seq_lens):
        return oracle_quant.kv_append_q8(k_codes, v_codes, k_scales, v_scales, k_new, v_new,
                                         block_table, np.asarray(seq_lens) + 1)

    return {
        "truncating": dict(quantize_rows_int8=truncating),
        "qmax_128": dict(QMAX=128),
        "scale_of_slot_zero": dict(gather_sequence_q8=scale_of_slot_zero),
        "no_scale": dict(dequantize_rows=no_scale),
        "swapped_kv_scales": dict(decode_attention_q8=swapped_kv_scales),
        "append_to_next_slot": dict(kv_append_q8=append_to_next_slot),
    }


@pytest.mark.parametrize("name", sorted(_mutants()))
def test_planted_mistake_is_caught(name):
    m = _mutant(**_mutants()[name])
    caught = (check_golden_rows(m) != 0 or check_golden_attend(m) > 1e-9
              or check_rounding_bound(m) != 0 or check_exact_reduces_to_fp16(m) > 0
              or check_append(m) != 0)
    assert caught, f"mutation {name} escaped every pin"
