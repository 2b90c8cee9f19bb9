"""Pins of the FP8 (E4M3) cache oracle (oracle/fp8.py) against what the
format definition, the quantisation rule and mathematics fix.  No GPU.

* Codes worked by hand from the E4M3 definition, and rows worked by hand
  (tests/golden/e4m3_rows.txt): values, ties to the even mantissa,
  subnormals, the sign of zero, and attention over dequantised rows.
* Every finite code round-trips, and the rounding agrees with PyTorch's own
  float8_e4m3fn conversion (a library routine) on random values and on every
  midpoint between neighbouring codes.
* The rounding bound: each code is within half a step of x / scale, and the
  largest magnitude of a nonzero row maps to +-448.
* A reduction to the fp16 oracle: when every value(code) * scale is exact in
  fp16, attention over the FP8 cache equals attention over that fp16 cache.
* Append: only the new slot changes.
A copy of the oracle with a planted mistake must fail at least one pin.
"""

from __future__ import annotations

import math
import os
import types

import numpy as np
import pytest

import oracle
from oracle import fp8 as oracle_fp8
from paged_kv_decode_24_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_rows.txt")


def _parse():
    codes, rows, attends, cur = {}, [], [], None
    with open(GOLDEN) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("code "):
                k, v = line[5:].split("=")
                codes[int(k, 16)] = float(v)
                continue
            if line.startswith("row ") or line.startswith("attend "):
                kind, name = line.split(None, 1)
                cur = {"name": name}
                (rows if kind == "row" else attends).append(cur)
                continue
            key, val = (x.strip() for x in line.split("=", 1))
            if key == "scale" and "math" in val:
                cur[key] = float(eval(val, {"math": math}))
            elif key == "scale" and "float32" in val:
                cur[key] = float(eval(val, {"float32": np.float32}))
            elif key == "scale":
                cur[key] = float(val)
            elif key in ("codes", "k_codes", "v_codes"):
                cur[key] = np.array([[int(x, 16) for x in r.split()] for r in val.split(";")],
                                    np.uint8)
            else:
                cur[key] = np.array([float(x) for x in val.split()])
    return codes, rows, attends


CODES, ROWS, ATTENDS = _parse()


# --------------------------------------------------------------------------
# checks, written against an oracle module so planted mistakes can be tried

def check_code_table(orc):
    bad = 0
    for c, v in CODES.items():
        got = float(orc.e4m3_value(np.array([c]))[0])
        bad += int(got != v or math.copysign(1.0, got) != math.copysign(1.0, v))
        bad += int(int(orc.e4m3_encode(np.array([v]))[0]) != c)
    bad += int(not np.isnan(orc.e4m3_value(np.array([0x7F, 0xFF]))).all())
    return bad


def check_roundtrip(orc):
    c = np.arange(256, dtype=np.uint8)
    v = orc.e4m3_value(c)
    fin = ~np.isnan(v)
    bad = int(np.sum(orc.e4m3_encode(v[fin]) != c[fin]))
    # finite values increase with the code within each sign
    pos = v[:0x7F]
    bad += int(np.sum(np.diff(pos) <= 0))
    return bad + int(fin.sum() != 254)


def check_against_torch(orc, seed=41):
    """Codes of random values and of every midpoint between neighbouring
    finite codes, against torch's float8_e4m3fn conversion."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(seed)
    vals = np.sort(orc.e4m3_value(np.arange(0x7F, dtype=np.uint8)))   # 0 .. 448
    mids = (vals[1:] + vals[:-1]) / 2
    xs = np.concatenate([rng.standard_normal(50000) * 40, rng.standard_normal(20000) * 0.01,
                         mids, -mids, vals, -vals]).astype(np.float32)
    xs = np.clip(xs, -448, 448)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return int(np.sum(orc.e4m3_encode(xs.astype(np.float64)) != want))


def check_golden_rows(orc):
    bad = 0
    for r in ROWS:
        x = r["x"].astype(np.float16)
        codes, scale = orc.quantize_rows_e4m3(x[None, :])
        bad += int(float(scale[0]) != r["scale"])
        bad += int(not np.array_equal(codes[0], r["codes"][0]))
    return bad


def check_golden_attend(orc):
    worst = 0.0
    S = 2
    for c in ATTENDS:
        L, D = c["k_codes"].shape
        pages = [int(p) for p in np.atleast_1d(c["pages"])]
        P = max(pages) + 1
        kc = np.full((P, 1, S, D), 0x7F, np.uint8)      # NaN codes outside the sequence
        vc = np.full((P, 1, S, D), 0xFF, np.uint8)
        ks = np.full((P, 1, S), 7.0, np.float32)
        vs = np.full((P, 1, S), 7.0, np.float32)
        for t in range(L):
            kc[pages[t // S], 0, t % S] = c["k_codes"][t]
            vc[pages[t // S], 0, t % S] = c["v_codes"][t]
            ks[pages[t // S], 0, t % S] = c["k_scales"][t]
            vs[pages[t // S], 0, t % S] = c["v_scales"][t]
        bt = np.array([pages], np.int32)
        got = orc.decode_attention_fp8(c["q"][None, None, :], kc, vc, ks, vs, bt, np.array([L]),
                                       c["scale"])
        worst = max(worst, float(np.max(np.abs(got[0, 0] - c["expect"]))))
    return worst


def check_rounding_bound(orc, seed=42):
    """Every code within half an E4M3 step of x / scale (relative 2^-4 for
    normals, 2^-10 absolute for subnormals), max |value| = 448 on nonzero
    rows, and scale = the nearest fp32 to amax / 448."""
    rng = np.random.default_rng(seed)
    bad = 0
    for sd in (1e-4, 0.02, 0.5, 3.0, 200.0):
        x = (rng.standard_normal((64, 128)) * sd).astype(np.float16)
        codes, scales = orc.quantize_rows_e4m3(x)
        xf = x.astype(np.float64)
        amax = np.abs(xf).max(axis=1)
        s64 = scales.astype(np.float64)
        ulp = np.spacing(scales).astype(np.float64)
        bad += int(np.sum(np.abs(s64 - amax / 448.0) > ulp / 2))
        ratio = xf / s64[:, None]
        val = orc.e4m3_value(codes)
        half_step = np.maximum(np.abs(ratio) * 2.0 ** -4, 2.0 ** -10)
        bad += int(np.sum(np.abs(ratio - val) > half_step * (1 + 1e-5)))
        bad += int(np.sum(np.abs(val).max(axis=1) != 448.0))
    return bad


def check_exact_reduces_to_fp16(orc, seed=43):
    """E4M3 values times power-of-two scales are exact in fp16: the FP8 oracle
    must equal the fp16 oracle on that fp16 cache, bit for bit."""
    rng = np.random.default_rng(seed)
    w = workloads.make_custom(seq_lens=[1, 19, 40, 16], num_q_heads=8, num_kv_heads=2,
                              head_dim=16, seed=44)
    shape = w.k_pages.shape
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    kc = rng.choice(finite, size=shape)
    vc = rng.choice(finite, size=shape)
    ks = np.ldexp(1.0, rng.integers(-8, 1, size=shape[:3])).astype(np.float32)
    vs = np.ldexp(1.0, rng.integers(-8, 1, size=shape[:3])).astype(np.float32)
    kp = (orc.e4m3_value(kc) * ks[..., None]).astype(np.float16)
    vp = (orc.e4m3_value(vc) * vs[..., None]).astype(np.float16)
    ref = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
    got = orc.decode_attention_fp8(w.q, kc, vc, ks, vs, w.block_table, w.seq_lens, w.scale)
    return float(np.max(np.abs(got - ref)))


def check_append(orc, seed=45):
    """Only the new slots change; they hold the new rows' codes; every other
    byte of the pools is untouched."""
    w = workloads.make_custom(seq_lens=[1, 16, 17, 40], num_q_heads=2, num_kv_heads=2,
                              head_dim=8, seed=seed)
    rng = np.random.default_rng(seed)
    shape = w.k_pages.shape
    kc = rng.integers(0, 256, size=shape).astype(np.uint8)
    vc = rng.integers(0, 256, size=shape).astype(np.uint8)
    ks = rng.random(shape[:3]).astype(np.float32)
    vs = rng.random(shape[:3]).astype(np.float32)
    kc2, vc2, ks2, vs2 = orc.kv_append_fp8(kc, vc, ks, vs, w.k_new, w.v_new, w.block_table,
                                           w.seq_lens)
    S = 16
    bad = 0
    touched = set()
    for b, L in enumerate(w.seq_lens):
        page, slot = int(w.block_table[b, (L - 1) // S]), (L - 1) % S
        touched.add((page, slot))
        for new, c2, s2 in ((w.k_new[b], kc2, ks2), (w.v_new[b], vc2, vs2)):
            deq = orc.e4m3_value(c2[page, :, slot]) * s2[page, :, slot, None].astype(np.float64)
            x = new.astype(np.float64)
            tol = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * s2[page, :, slot, None]) * 1.0001
            bad += int(np.sum(np.abs(deq - x) > tol))
    for (a, a2) in ((kc, kc2), (vc, vc2), (ks, ks2), (vs, vs2)):
        diff = np.argwhere(np.any((a != a2).reshape(shape[0], shape[1], S, -1), axis=(1, 3)))
        bad += len(set((int(p), int(s)) for p, s in diff) - touched)
    return bad


# --------------------------------------------------------------------------
# the pins

def test_code_table_from_the_format_definition():
    assert check_code_table(oracle) == 0


def test_every_finite_code_round_trips():
    assert check_roundtrip(oracle) == 0


def test_rounding_matches_torch_float8():
    assert check_against_torch(oracle) == 0


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


def test_saturation_and_zero_row():
    assert list(oracle.e4m3_round(np.array([470.0, -1e6, 463.9]))) == [448.0, -448.0, 448.0]
    codes, scales = oracle.quantize_rows_e4m3(np.zeros((3, 16), np.float16))
    assert np.all(codes == 0) and np.all(scales == 0)
    w = workloads.make_custom(seq_lens=[0, 3], num_q_heads=2, num_kv_heads=1, head_dim=8, seed=46)
    shape = w.k_pages.shape
    kc = np.full(shape, 0x38, np.uint8)          # every value 1.0
    ks = np.ones(shape[:3], np.float32)
    got = oracle.decode_attention_fp8(w.q, kc, kc, ks, ks, w.block_table, w.seq_lens, w.scale)
    assert np.all(got[0] == 0.0)
    np.testing.assert_allclose(got[1], 1.0, rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# planted mistakes

def _mutant(**overrides):
    m = types.ModuleType("oracle_fp8_mutant")
    m.__dict__.update(vars(oracle_fp8))
    m.__dict__.update(overrides)
    for name, fn in list(m.__dict__.items()):
        if isinstance(fn, types.FunctionType) and name not in overrides:
            m.__dict__[name] = types.FunctionType(fn.__code__, m.__dict__, name, fn.__defaults__)
    return m


def _mutants():
    def ties_away(x):
        x = np.asarray(x, np.float64)
        a = np.minimum(np.abs(x), 448.0)
        _, k = np.frexp(np.where(a >= 2.0 ** -6, a, 2.0 ** -6))
        step = np.where(a >= 2.0 ** -6, np.ldexp(1.0, k - 4), 2.0 ** -9)
        return np.copysign(np.minimum(np.floor(a / step + 0.5) * step, 448.0), x)

    def truncating(x):
        x = np.asarray(x, np.float64)
        a = np.minimum(np.abs(x), 448.0)
        _, k = np.frexp(np.where(a >= 2.0 ** -6, a, 2.0 ** -6))
        step = np.where(a >= 2.0 ** -6, np.ldexp(1.0, k - 4), 2.0 ** -9)
        return np.copysign(np.floor(a / step) * step, x)

    def flush_subnormals(codes):
        v = oracle_fp8.e4m3_value(codes)
        return np.where(np.abs(v) < 2.0 ** -6, 0.0, v)

    def scale_of_slot_zero(codes, scales, block_table, b, seq_len, kv_head):
        S = codes.shape[2]
        t = np.arange(seq_len)
        phys = block_table[b, t // S].astype(np.int64)
        return oracle_fp8.e4m3_value(codes[phys, kv_head, t % S, :]) * \
            scales[phys, kv_head, 0].astype(np.float64)[:, None]

    def swapped_kv_scales(q, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens, scale,
                          heads=None):
        return oracle_fp8.decode_attention_fp8(q, k_codes, v_codes, v_scales, k_scales,
                                               block_table, seq_lens, scale, heads)

    def append_to_next_slot(k_codes, v_codes, k_scales, v_scales, k_new, v_new, block_table,
                            seq_lens):
        return oracle_fp8.kv_append_fp8(k_codes, v_codes, k_scales, v_scales, k_new, v_new,
                                        block_table, np.asarray(seq_lens) + 1)

    return {
        "ties_away_from_zero": dict(e4m3_round=ties_away),
        "truncating": dict(e4m3_round=truncating),
        "bias_8": dict(E4M3_BIAS=8),
        "max_240": dict(E4M3_MAX=240.0),
        "flush_subnormals": dict(e4m3_value=flush_subnormals),
        "scale_of_slot_zero": dict(gather_sequence_fp8=scale_of_slot_zero),
        "swapped_kv_scales": dict(decode_attention_fp8=swapped_kv_scales),
        "append_to_next_slot": dict(kv_append_fp8=append_to_next_slot),
    }


@pytest.mark.parametrize("name", sorted(_mutants()))
def test_planted_mistake_is_caught(name):
    m = _mutant(**_mutants()[name])
    caught = (check_code_table(m) != 0 or check_roundtrip(m) != 0 or check_golden_rows(m) != 0
              or check_golden_attend(m) > 1e-9 or check_rounding_bound(m) != 0
              or check_exact_reduces_to_fp16(m) > 0 or check_append(m) != 0)
    assert caught, f"mutation {name} escaped every pin"
