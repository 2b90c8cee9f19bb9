"""Oracle for decode attention over an INT8 paged KV cache.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module; the library never does, and this module
imports nothing from the library.

What it computes, and where the pages define it:

* KV-cache quantisation -- MonadKai/xLLM, introduction: the KV cache supports
  quantisation, and the quantisation list names per-row INT8.
* Everything after dequantisation is the fp16 oracle in ``attention.py``:
  the same gather through the block table and the same float64 softmax
  attention.

Readings of what the pages leave open:

* A row is one token's D-vector of one KV head: the (page, kv_head, slot)
  row of the pool.  Each row has its own scale.
* Quantisation is symmetric: scale = max|x| / 127, code = x / scale rounded
  to nearest, ties to even, clamped to [-127, 127].  An all-zero row has
  scale 0 and all-zero codes.
* Those three steps take integer decisions, so they are done in IEEE fp32
  (numpy float32: correctly rounded division, then round-half-even), the
  precision the kernel uses.  Any implementation that divides in fp32 picks
  the same codes.
* The dequantised value is code * scale, taken exactly in float64.
* Codes sit in a pool [page][kv_head][slot][dim] int8, scales in a pool
  [page][kv_head][slot] float32.
"""

from __future__ import annotations

import numpy as np

from .attention import attend_one

QMAX = 127


def quantize_rows_int8(x: np.ndarray):
    """Per-row symmetric INT8 codes and fp32 scales of the last axis of ``x``.

    Returns (codes int8 [..., D], scales float32 [...]).
    """
    x32 = np.asarray(x).astype(np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    scales = (amax / np.float32(QMAX)).astype(np.float32)
    safe = np.where(scales > 0, scales, np.float32(1.0)).astype(np.float32)
    ratio = (x32 / safe[..., None]).astype(np.float32)
    codes = np.clip(np.rint(ratio), -QMAX, QMAX)
    codes = np.where(scales[..., None] > 0, codes, 0.0)
    return codes.astype(np.int8), scales


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """code * scale in float64 (exact: an int8 times an fp32 fits in a double)."""
    return codes.astype(np.float64) * scales.astype(np.float64)[..., None]


def gather_sequence_q8(codes, scales, block_table, b, seq_len, kv_head):
    """Dequantised logical [L][D] float64 rows of one sequence and KV head."""
    S = codes.shape[2]
    t = np.arange(seq_len)
    phys = block_table[b, t // S].astype(np.int64)
    return dequantize_rows(codes[phys, kv_head, t % S, :], scales[phys, kv_head, t % S])


def kv_append_q8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, block_table, seq_lens):
    """Quantise the new token's K and V rows and write codes and scales at
    logical position L_b - 1.  Returns new pools; the inputs are untouched."""
    kc, vc = k_codes.copy(), v_codes.copy()
    ks, vs = k_scales.copy(), v_scales.copy()
    S = k_codes.shape[2]
    new_kc, new_ks = quantize_rows_int8(k_new)   # [B][Hkv][D], [B][Hkv]
    new_vc, new_vs = quantize_rows_int8(v_new)
    for b in range(len(seq_lens)):
        pos = int(seq_lens[b]) - 1
        if pos < 0:
            continue
        page = int(block_table[b, pos // S])
        kc[page, :, pos % S, :] = new_kc[b]
        vc[page, :, pos % S, :] = new_vc[b]
        ks[page, :, pos % S] = new_ks[b]
        vs[page, :, pos % S] = new_vs[b]
    return kc, vc, ks, vs


def decode_attention_q8(q, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens, scale,
                        heads=None):
    """Decode attention over the dequantised cache, float64 [B][Hq][D].

    ``heads``, if given, lists the (b, h) pairs to compute; others stay NaN.
    """
    B, Hq, D = q.shape
    Hkv = k_codes.shape[1]
    G = Hq // Hkv
    out = np.full((B, Hq, D), np.nan, np.float64)
    wanted = None if heads is None else set((int(b), int(h)) for b, h in heads)
    for b in range(B):
        L = int(seq_lens[b])
        for g in range(Hkv):
            hs = [h for h in range(g * G, (g + 1) * G) if wanted is None or (b, h) in wanted]
            if not hs:
                continue
            K = gather_sequence_q8(k_codes, k_scales, block_table, b, L, g)
            V = gather_sequence_q8(v_codes, v_scales, block_table, b, L, g)
            for h in hs:
                out[b, h] = attend_one(q[b, h], K, V, scale)
    return out
