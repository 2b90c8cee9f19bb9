"""Pins of the float64 oracle against what the definition and mathematics fix.

No GPU.  Every pin compares the oracle with something other than itself:
hand-derived closed forms (tests/golden/), a brute-force route that builds the
contiguous cache first and scatters it into pages, special cases that reduce
to a mean or a single row, invariances of softmax attention, and the
log-sum-exp split identity.  ``check_*`` helpers take the oracle module as an
argument so the mutation test at the bottom can run them on a copy of the
oracle with a planted mistake and see them fail.
"""

from __future__ import annotations

import math
import os
import types

import numpy as np
import pytest

import oracle
from oracle import attention as oracle_attention
from paged_kv_decode_24_gb300 import accounting, workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# brute force: contiguous cache first, scattered into pages afterwards

def dense_case(rng, B, Hq, Hkv, D, S, lens, pool_pages=None):
    """Contiguous per-sequence K/V, scattered into a paged pool by a route
    independent of the oracle: a python loop over tokens with an explicit
    (page, slot) table."""
    pages_needed = [(L + S - 1) // S for L in lens]
    P = pool_pages or max(1, sum(pages_needed) + 3)
    perm = rng.permutation(P)
    bt = np.full((B, max(max(pages_needed), 1)), -1, np.int32)
    cur = 0
    for b, n in enumerate(pages_needed):
        bt[b, :n] = perm[cur:cur + n]
        cur += n
    dense_k = [rng.standard_normal((Hkv, L, D)) for L in lens]
    dense_v = [rng.standard_normal((Hkv, L, D)) for L in lens]
    kp = rng.standard_normal((P, Hkv, S, D)) * 1e3   # junk everywhere first
    vp = rng.standard_normal((P, Hkv, S, D)) * 1e3
    slots = {}
    for b, L in enumerate(lens):
        for t in range(L):
            page, slot = int(bt[b, t // S]), t % S
            slots[(b, t)] = page * S + slot
            kp[page, :, slot, :] = dense_k[b][:, t, :]
            vp[page, :, slot, :] = dense_v[b][:, t, :]
    q = rng.standard_normal((B, Hq, D))
    return q, kp, vp, bt, np.array(lens, np.int32), dense_k, dense_v, slots


def brute_force(q, dense_k, dense_v, lens, scale, G):
    """Naive attention with python floats, no max shift (inputs are small)."""
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            w = [math.exp(scale * math.fsum(q[b, h, d] * dense_k[b][g, t, d] for d in range(D)))
                 for t in range(lens[b])]
            tot = math.fsum(w)
            for d in range(D):
                out[b, h, d] = math.fsum(w[t] * dense_v[b][g, t, d] for t in range(lens[b])) / tot \
                    if lens[b] else 0.0
    return out


def check_brute_force(orc, seed=1):
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, D, S = 3, 4, 2, 8, 4
    lens = [5, 1, 11]
    q, kp, vp, bt, sl, dk, dv, _ = dense_case(rng, B, Hq, Hkv, D, S, lens)
    scale = 0.37
    got = orc.decode_attention(q, kp, vp, bt, sl, scale)
    want = brute_force(q, dk, dv, lens, scale, Hq // Hkv)
    return np.max(np.abs(got - want))


def check_gather_slots(orc, seed=2):
    rng = np.random.default_rng(seed)
    lens = [7, 0, 16, 33]
    q, kp, vp, bt, sl, dk, dv, slots = dense_case(rng, 4, 2, 2, 4, 8, lens)
    got = orc.gather_slots(bt, sl, 8)
    bad = 0
    for b, L in enumerate(lens):
        for t in range(got.shape[1]):
            want = slots[(b, t)] if t < L else -1
            bad += int(got[b, t] != want)
    return bad


def check_split_equals_unsplit(orc, seed=3):
    rng = np.random.default_rng(seed)
    lens = [1, 17, 64, 45]
    q, kp, vp, bt, sl, *_ = dense_case(rng, 4, 4, 1, 16, 8, lens)
    ref = orc.decode_attention(q, kp, vp, bt, sl, 0.25)
    worst = 0.0
    for chunk in (1, 2, 3, 8):
        got = orc.decode_attention_split(q, kp, vp, bt, sl, 0.25, chunk)
        worst = max(worst, float(np.max(np.abs(got - ref))))
    return worst


# --------------------------------------------------------------------------
# the pins

def test_brute_force_tiny():
    assert check_brute_force(oracle) < 1e-12


def test_gather_slots_exact():
    assert check_gather_slots(oracle) == 0


def test_split_equals_unsplit():
    assert check_split_equals_unsplit(oracle) < 1e-13


def _parse_golden():
    cases = []
    cur = None
    with open(os.path.join(GOLDEN, "softmax_closed_form.txt")) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("case "):
                cur = {"name": line[5:]}
                cases.append(cur)
                continue
            key, val = (x.strip() for x in line.split("=", 1))
            val = val.replace("LN2", repr(math.log(2))).replace("LN5", repr(math.log(5)))
            if key == "scale":
                cur[key] = float(eval(val, {"math": math}))
            elif key in ("K", "V"):
                cur[key] = np.array([[float(x) for x in row.split()] for row in val.split(";")])
            elif key == "pages":
                cur[key] = [int(x) for x in val.split()]
            else:
                cur[key] = np.array([float(x) for x in val.split()])
    return cases


@pytest.mark.parametrize("case", _parse_golden(), ids=lambda c: c["name"])
def test_golden_closed_form(case):
    K, V, pages = case["K"], case["V"], case["pages"]
    S, D = 2, K.shape[1]
    L = K.shape[0]
    P = max(pages) + 1
    kp = np.full((P, 1, S, D), 7.0)
    vp = np.full((P, 1, S, D), 7.0)
    for t in range(L):
        kp[pages[t // S], 0, t % S] = K[t]
        vp[pages[t // S], 0, t % S] = V[t]
    bt = np.array([pages], np.int32)
    got = oracle.decode_attention(case["q"][None, None, :], kp, vp, bt, np.array([L]), case["scale"])
    np.testing.assert_allclose(got[0, 0], case["expect"], rtol=0, atol=1e-12)


def test_uniform_scores_give_mean_of_v():
    rng = np.random.default_rng(4)
    q, kp, vp, bt, sl, dk, dv, _ = dense_case(rng, 2, 2, 1, 8, 4, [9, 30])
    q[:] = 0.0
    got = oracle.decode_attention(q, kp, vp, bt, sl, 1.0)
    for b in range(2):
        np.testing.assert_allclose(got[b, 0], dv[b][0].mean(axis=0), rtol=0, atol=1e-13)


def test_equal_keys_give_mean_of_v():
    rng = np.random.default_rng(5)
    q, kp, vp, bt, sl, dk, dv, _ = dense_case(rng, 1, 1, 1, 8, 4, [13])
    row = rng.standard_normal(8)
    for t in range(13):
        kp[bt[0, t // 4], 0, t % 4] = row
    got = oracle.decode_attention(q, kp, vp, bt, sl, 0.9)
    np.testing.assert_allclose(got[0, 0], dv[0][0].mean(axis=0), rtol=0, atol=1e-13)


@pytest.mark.parametrize("D,t_star", [(64, 0), (64, 99), (128, 50)])
def test_one_hot_selects_row(D, t_star):
    rng = np.random.default_rng(6)
    L = 100
    q, kp, vp, bt, sl, dk, dv, _ = dense_case(rng, 1, 1, 1, D, 16, [L])
    q[:] = 0.0
    q[0, 0, 0] = 16.0
    for t in range(L):
        kp[bt[0, t // 16], 0, t % 16, 0] = 16.0 if t == t_star else 0.0
    scale = 1.0 / math.sqrt(D)
    gap = 256.0 * scale
    got = oracle.decode_attention(q, kp, vp, bt, sl, scale)[0, 0]
    bound = L * math.exp(-gap) * 2 * np.abs(dv[0][0]).max()
    assert np.max(np.abs(got - dv[0][0][t_star])) <= bound


def test_seq_len_one_is_exact_v0():
    rng = np.random.default_rng(7)
    q, kp, vp, bt, sl, dk, dv, _ = dense_case(rng, 3, 4, 2, 16, 16, [1, 1, 1])
    got = oracle.decode_attention(q, kp, vp, bt, sl, 0.3)
    for b in range(3):
        for h in range(4):
            assert np.array_equal(got[b, h], dv[b][h // 2][0])


def test_seq_len_zero_is_zero():
    rng = np.random.default_rng(8)
    q, kp, vp, bt, sl, *_ = dense_case(rng, 2, 2, 2, 8, 4, [0, 5])
    got = oracle.decode_attention(q, kp, vp, bt, sl, 0.3)
    assert np.all(got[0] == 0.0)
    assert np.all(np.isfinite(got[1]))


def test_page_permutation_invariance():
    """Relabelling physical pages (and rewriting the block table) changes nothing."""
    w = workloads.make_custom(seq_lens=[37, 100, 5], num_q_heads=4, num_kv_heads=2,
                              head_dim=64, num_pages=40, dist=("uniform", 1.0), seed=9)
    ref = oracle.decode_attention(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens, w.scale)
    perm = np.random.default_rng(10).permutation(w.num_pages)
    kp = np.empty_like(w.k_pages)
    vp = np.empty_like(w.v_pages)
    kp[perm] = w.k_pages
    vp[perm] = w.v_pages
    bt = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    got = oracle.decode_attention(w.q, kp, vp, bt, w.seq_lens, w.scale)
    assert np.array_equal(got, ref)


def test_gqa_equals_mha_with_repeated_heads():
    w = workloads.make_custom(seq_lens=[20, 49], num_q_heads=8, num_kv_heads=2, head_dim=16,
                              seed=11)
    ref = oracle.decode_attention(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens, w.scale)
    kp = np.repeat(w.k_pages, 4, axis=1)   # KV head g becomes query heads 4g..4g+3
    vp = np.repeat(w.v_pages, 4, axis=1)
    got = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-14)


def test_affine_in_v():
    rng = np.random.default_rng(12)
    q, kp, vp, bt, sl, *_ = dense_case(rng, 2, 2, 2, 8, 4, [6, 21])
    base = oracle.decode_attention(q, kp, vp, bt, sl, 0.5)
    alpha, c = -2.5, 3.25
    got = oracle.decode_attention(q, kp, alpha * vp + c, bt, sl, 0.5)
    np.testing.assert_allclose(got, alpha * base + c, rtol=0, atol=1e-12)


def test_kv_append_writes_only_the_new_slot():
    w = workloads.make_custom(seq_lens=[1, 16, 17, 40], num_q_heads=2, num_kv_heads=2,
                              head_dim=8, seed=13)
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    slots = oracle.gather_slots(w.block_table, w.seq_lens, 16)
    changed = np.argwhere(np.any(kp.view(np.uint16) != w.k_pages.view(np.uint16), axis=(1, 3)))
    S = 16
    written = sorted((int(slots[b, L - 1]) // S, int(slots[b, L - 1]) % S)
                     for b, L in enumerate(w.seq_lens))
    for (page, slot) in written:
        b = [i for i, L in enumerate(w.seq_lens) if slots[i, L - 1] == page * S + slot][0]
        assert np.array_equal(kp[page, :, slot].view(np.uint16), w.k_new[b].view(np.uint16))
        assert np.array_equal(vp[page, :, slot].view(np.uint16), w.v_new[b].view(np.uint16))
    assert sorted(set((int(p), int(s)) for p, s in changed)) == sorted(set(written))


def test_fp16_inputs_widen_exactly():
    """Output of a one-token sequence equals the fp16 V row bit for bit after
    widening, so no precision is lost on the way in."""
    w = workloads.make_custom(seq_lens=[1], num_q_heads=1, num_kv_heads=1, head_dim=64, seed=14)
    got = oracle.decode_attention(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens, w.scale)
    row = w.v_pages[w.block_table[0, 0], 0, 0].astype(np.float64)
    assert np.array_equal(got[0, 0], row)


def test_kv_cache_memory_formula_matches_xllm_table():
    vals = {}
    with open(os.path.join(GOLDEN, "kv_cache_memory.txt")) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                k, v = (x.strip() for x in line.split("="))
                vals[k] = int(v)
    n_bytes = accounting.kv_cache_bytes([vals["s"] + vals["n"]] * vals["b"], vals["h1"],
                                        vals["bytes_per_element"], layers=vals["layers"],
                                        round_to=vals["round_to"])
    assert n_bytes == vals["expect_gib"] * 2**30


# --------------------------------------------------------------------------
# planted mistakes: each mutated copy of the oracle must fail at least one pin

def _mutant(**overrides):
    src = dict(vars(oracle_attention))
    m = types.ModuleType("oracle_mutant")
    m.__dict__.update(src)
    m.__dict__.update(overrides)
    # make functions resolve globals in the mutant
    for name, fn in list(m.__dict__.items()):
        if isinstance(fn, types.FunctionType) and name not in overrides:
            m.__dict__[name] = types.FunctionType(fn.__code__, m.__dict__, name, fn.__defaults__)
    return m


def _mutants():
    np_ = np

    def gqa_modulo(q, k_pages, v_pages, block_table, seq_lens, scale, heads=None):
        B, Hq, D = q.shape
        Hkv = k_pages.shape[1]
        out = np_.zeros((B, Hq, D))
        for b in range(B):
            for h in range(Hq):
                K = oracle_attention.gather_sequence(k_pages, block_table, b, int(seq_lens[b]), h % Hkv)
                V = oracle_attention.gather_sequence(v_pages, block_table, b, int(seq_lens[b]), h % Hkv)
                out[b, h] = oracle_attention.attend_one(q[b, h], K, V, scale)
        return out

    def slot_transposed(pages, block_table, b, seq_len, kv_head):
        S = pages.shape[2]
        t = np_.arange(seq_len)
        return pages[block_table[b, t % S] if False else block_table[b, t // S], kv_head,
                     (S - 1 - t % S), :].astype(np_.float64)

    def no_scale(q_row, keys, values, scale):
        s = keys @ q_row.astype(np_.float64)
        e = np_.exp(s - s.max())
        return (e / e.sum()) @ values if keys.shape[0] else np_.zeros(values.shape[1])

    def drop_last_token(pages, block_table, b, seq_len, kv_head):
        return oracle_attention.gather_sequence(pages, block_table, b, max(seq_len - 1, 1), kv_head)

    def sign_flip(q_row, keys, values, scale):
        s = -scale * (keys @ q_row.astype(np_.float64))
        e = np_.exp(s - s.max())
        return (e / e.sum()) @ values if keys.shape[0] else np_.zeros(values.shape[1])

    def lse_wrong(q_row, keys, values, scale):
        o, lse = oracle_attention.split_partial(q_row, keys, values, scale)
        return o, lse - np_.log(max(keys.shape[0], 1))

    def slots_off_by_one(block_table, seq_lens, page_size):
        out = oracle_attention.gather_slots(block_table, seq_lens, page_size)
        out[out >= 0] += 1
        return out

    return {
        "gqa_modulo": dict(decode_attention=gqa_modulo),
        "slot_reversed": dict(gather_sequence=slot_transposed),
        "no_scale": dict(attend_one=no_scale),
        "drop_last_token": dict(gather_sequence=drop_last_token),
        "sign_flip": dict(attend_one=sign_flip),
        "lse_wrong": dict(split_partial=lse_wrong),
        "slots_off_by_one": dict(gather_slots=slots_off_by_one),
    }


@pytest.mark.parametrize("name", sorted(_mutants()))
def test_planted_mistake_is_caught(name):
    m = _mutant(**_mutants()[name])
    caught = (check_brute_force(m) > 1e-9 or check_gather_slots(m) != 0
              or check_split_equals_unsplit(m) > 1e-9)
    assert caught, f"mutation {name} escaped every pin"
