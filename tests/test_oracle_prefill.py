"""Pins of the multi-token oracle (oracle/prefill.py).  No GPU.

* One query token per sequence reduces to the decode oracle.
* A whole prompt (q_lens = L) equals textbook causal attention over the
  contiguous sequence, written as masked matrix products.
* A brute force with python floats on tiny mixed batches.
* Causality: changing keys and values after a query's position leaves its
  output unchanged, bit for bit.
* The multi-row append writes exactly the new rows at the newest positions.
Planted mistakes in a copy of the oracle must fail one of these.
"""

from __future__ import annotations

import math
import types

import numpy as np
import pytest

import oracle
from oracle import attention as oracle_attention
from oracle import prefill as oracle_prefill
from paged_kv_decode_24_gb300 import workloads


def _case(lens, q_lens, hq=4, hkv=2, d=16, seed=0, dist=("normal", 0.5)):
    return workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                 seed=seed, q_lens=q_lens, dist=dist)


def check_reduces_to_decode(orc):
    w = _case([5, 37, 100, 16], [1, 1, 1, 1], seed=81)
    got = orc.prefill_attention(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens, w.q_lens,
                                w.scale)
    want = oracle.decode_attention(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens, w.scale)
    return float(np.max(np.abs(got - want)))


def check_full_prompt_is_causal_attention(orc):
    lens = [23, 40]
    w = _case(lens, lens, hq=4, hkv=2, d=8, seed=82)
    got = orc.prefill_attention(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens, w.q_lens,
                                w.scale)
    worst = 0.0
    cu = np.concatenate([[0], np.cumsum(lens)])
    for b, L in enumerate(lens):
        for h in range(4):
            g = h // 2
            K = np.stack([w.k_pages[w.block_table[b, t // 16], g, t % 16] for t in range(L)]).astype(np.float64)
            V = np.stack([w.v_pages[w.block_table[b, t // 16], g, t % 16] for t in range(L)]).astype(np.float64)
            Q = w.q[cu[b]:cu[b + 1], h].astype(np.float64)
            S = w.scale * Q @ K.T
            S[np.triu_indices(L, 1)] = -np.inf
            P = np.exp(S - S.max(axis=1, keepdims=True))
            O = (P / P.sum(axis=1, keepdims=True)) @ V
            worst = max(worst, float(np.max(np.abs(O - got[cu[b]:cu[b + 1], h]))))
    return worst


def check_brute_force(orc):
    lens, qls = [9, 4, 20], [3, 4, 1]
    w = _case(lens, qls, hq=2, hkv=1, d=4, seed=83)
    got = orc.prefill_attention(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens, w.q_lens,
                                w.scale)
    worst, r = 0.0, 0
    for b, (L, n) in enumerate(zip(lens, qls)):
        for i in range(n):
            p = L - n + i
            for h in range(2):
                ks = [[float(x) for x in w.k_pages[w.block_table[b, t // 16], 0, t % 16]]
                      for t in range(p + 1)]
                vs = [[float(x) for x in w.v_pages[w.block_table[b, t // 16], 0, t % 16]]
                      for t in range(p + 1)]
                qv = [float(x) for x in w.q[r, h]]
                e = [math.exp(w.scale * math.fsum(a * c for a, c in zip(qv, k))) for k in ks]
                z = math.fsum(e)
                o = [math.fsum(e[t] * vs[t][d] for t in range(p + 1)) / z for d in range(4)]
                worst = max(worst, max(abs(o[d] - got[r, h, d]) for d in range(4)))
            r += 1
    return worst


def check_causality(orc):
    w = _case([50], [10], hq=2, hkv=1, d=8, seed=84)
    base = orc.prefill_attention(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens, w.q_lens,
                                 w.scale)
    kp, vp = w.k_pages.copy(), w.v_pages.copy()
    for t in range(45, 50):                     # positions of queries 5..9
        kp[w.block_table[0, t // 16], 0, t % 16] += np.float16(3.0)
        vp[w.block_table[0, t // 16], 0, t % 16] -= np.float16(2.0)
    got = orc.prefill_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.q_lens, w.scale)
    same = np.array_equal(got[:5], base[:5])
    changed = not np.allclose(got[5:], base[5:])
    return same and changed


def check_append(orc):
    w = _case([3, 17, 40, 16], [3, 2, 17, 0], seed=85)
    kp, vp = orc.kv_append_tokens(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                  w.seq_lens, w.q_lens)
    bad = 0
    r = 0
    written = set()
    for b, (L, n) in enumerate(zip(w.seq_lens, w.q_lens)):
        for i in range(n):
            t = L - n + i
            page, slot = int(w.block_table[b, t // 16]), t % 16
            written.add((page, slot))
            bad += int(not np.array_equal(kp[page, :, slot], w.k_new[r]))
            bad += int(not np.array_equal(vp[page, :, slot], w.v_new[r]))
            r += 1
    diff = np.argwhere(np.any(kp.view(np.uint16) != w.k_pages.view(np.uint16), axis=(1, 3)))
    bad += len(set((int(p), int(s)) for p, s in diff) - written)
    return bad


def test_reduces_to_decode():
    assert check_reduces_to_decode(oracle) == 0.0


def test_full_prompt_is_causal_attention():
    assert check_full_prompt_is_causal_attention(oracle) < 1e-13


def test_brute_force_tiny():
    assert check_brute_force(oracle) < 1e-12


def test_causality():
    assert check_causality(oracle)


def test_append_writes_only_the_new_rows():
    assert check_append(oracle) == 0
    w = _case([3, 17, 40], [1, 1, 1], seed=86)
    a = oracle.kv_append_tokens(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                w.seq_lens, w.q_lens)
    b = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_empty_query_sets():
    w = _case([0, 5, 12], [0, 0, 4], seed=87)
    got = oracle.prefill_attention(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens,
                                   w.q_lens, w.scale)
    assert got.shape[0] == 4 and np.all(np.isfinite(got))


def _mutant(**overrides):
    m = types.ModuleType("oracle_prefill_mutant")
    m.__dict__.update(vars(oracle_prefill))
    m.__dict__.update(overrides)
    for name, fn in list(m.__dict__.items()):
        if isinstance(fn, types.FunctionType) and name not in overrides:
            m.__dict__[name] = types.FunctionType(fn.__code__, m.__dict__, name, fn.__defaults__)
    return m


def _mutants():
    def strict_causal(q_row, keys, values, scale):
        return oracle_attention.attend_one(q_row, keys[:-1] if len(keys) > 1 else keys,
                                           values[:-1] if len(values) > 1 else values, scale)

    def gather_from_zero(pages, block_table, b, seq_len, kv_head):
        # positions counted from the first query instead of the sequence start
        full = oracle_attention.gather_sequence(pages, block_table, b, seq_len, kv_head)
        return np.concatenate([full[1:], full[:1]])

    def append_one_late(k_pages, v_pages, k_new, v_new, block_table, seq_lens, q_lens):
        return oracle_prefill.kv_append_tokens(k_pages, v_pages, k_new, v_new, block_table,
                                               np.asarray(seq_lens) + 1, q_lens)

    return {"strict_causal": dict(attend_one=strict_causal),
            "shifted_positions": dict(gather_sequence=gather_from_zero),
            "append_one_late": dict(kv_append_tokens=append_one_late)}


@pytest.mark.parametrize("name", sorted(_mutants()))
def test_planted_mistake_is_caught(name):
    m = _mutant(**_mutants()[name])
    try:
        caught = (check_reduces_to_decode(m) > 1e-9 or check_full_prompt_is_causal_attention(m) > 1e-9
                  or check_brute_force(m) > 1e-9 or not check_causality(m) or check_append(m) != 0)
    except (IndexError, ValueError):
        caught = True
    assert caught, f"mutation {name} escaped every pin"
