"""Oracle for decode attention over an FP8 (E4M3) paged KV cache.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module; the library never does, and this module
imports nothing from the library.

What it computes, and where the pages define it:

* KV-cache quantisation -- MonadKai/xLLM, introduction (the KV cache supports
  quantisation); "Eine LLM-Inferenz-Engine von Grund auf mit C++ und CUDA
  bauen", section 4 (future directions: stronger quantisation, FP8, INT8 or
  INT4, of activations and the cache).
* Everything after dequantisation is the fp16 oracle in ``attention.py``:
  the same gather through the block table and the same float64 softmax
  attention.

Readings of what the pages leave open:

* FP8 is the E4M3 format of the OCP 8-bit floating-point specification: a
  sign bit, four exponent bits with bias 7 and three mantissa bits.  An
  exponent field of 0 holds the subnormals m/8 * 2^-6; there are no
  infinities; S.1111.111 is NaN, so the largest finite magnitude is
  1.75 * 2^8 = 448 (S.1111.110).
* As for the INT8 cache, a row is one token's D-vector of one KV head and has
  its own fp32 scale: scale = max|x| / 448, and code = E4M3 of x / scale,
  rounded to the nearest E4M3 value with ties to the even mantissa, any
  magnitude above 448 clamped to 448 (the ratio of the largest element can
  exceed 448 by an fp32 rounding).  An all-zero row has scale 0 and zero
  codes.
* Both divisions take the decisions that fix the codes, so they are done in
  IEEE fp32 (numpy float32, correctly rounded), the precision the kernel
  uses; the rounding to E4M3 is then exact arithmetic on that fp32 ratio.
* The dequantised value is value(code) * scale, exact in float64.
* Codes sit in a pool [page][kv_head][slot][dim] of bytes (uint8), scales in
  a pool [page][kv_head][slot] float32.
"""

from __future__ import annotations

import numpy as np

from .attention import attend_one

E4M3_MAX = 448.0
E4M3_BIAS = 7
MIN_NORMAL = 2.0 ** -6       # exponent field 1, mantissa 0
SUBNORMAL_STEP = 2.0 ** -9   # mantissa step of the subnormals (exponent field 0)


def e4m3_value(codes) -> np.ndarray:
    """The float64 value of each E4M3 byte (NaN for S.1111.111)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - E4M3_BIAS).astype(np.int64))
    sub = m * SUBNORMAL_STEP
    v = sign * np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def e4m3_round(x) -> np.ndarray:
    """Nearest E4M3 value to each finite x (ties to the even mantissa), with
    magnitudes above 448 clamped to 448; float64 in, float64 out."""
    x = np.asarray(x, np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # the spacing of the grid a falls on: 2^-9 below 2^-6, else 2^(e-3) for
    # a in [2^e, 2^(e+1)) (frexp gives a = f * 2^k with f in [0.5, 1): e = k-1)
    _, k = np.frexp(np.where(a >= MIN_NORMAL, a, MIN_NORMAL))
    step = np.where(a >= MIN_NORMAL, np.ldexp(1.0, k - 4), SUBNORMAL_STEP)
    # a / step is exact (a power-of-two step); rint rounds half to even, so a
    # tie goes to the even count of steps, i.e. the even mantissa
    r = np.rint(a / step) * step
    return np.copysign(np.minimum(r, E4M3_MAX), x)


def e4m3_encode(x) -> np.ndarray:
    """The E4M3 byte of each value of ``e4m3_round(x)``, keeping the sign of x."""
    v = e4m3_round(x)
    a = np.abs(v)
    sign = np.where(np.signbit(v), 0x80, 0)  # the sign of x, a zero's too (as IEEE conversions do)
    sub = a < MIN_NORMAL
    f, k = np.frexp(np.where(sub, 1.0, a))          # a = (2f) * 2^(k-1), 2f in [1, 2)
    e = np.where(sub, 0, k - 1 + E4M3_BIAS).astype(np.int64)
    m = np.where(sub, a / SUBNORMAL_STEP, (2.0 * f - 1.0) * 8.0)   # exact small integers
    return (sign | (e << 3) | m.astype(np.int64)).astype(np.uint8)


def quantize_rows_e4m3(x: np.ndarray):
    """Per-row E4M3 codes and fp32 scales of the last axis of ``x``.

    Returns (codes uint8 [..., D], scales float32 [...]).
    """
    x32 = np.asarray(x).astype(np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    scales = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scales > 0, scales, np.float32(1.0)).astype(np.float32)
    ratio = (x32 / safe[..., None]).astype(np.float32)
    codes = e4m3_encode(ratio.astype(np.float64))
    codes = np.where(scales[..., None] > 0, codes, 0).astype(np.uint8)
    return codes, scales


def dequantize_rows_e4m3(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """value(code) * scale in float64 (exact: 4 significant bits times an fp32).
    The values of the 256 bytes are listed once per call and looked up."""
    table = e4m3_value(np.arange(256, dtype=np.uint8))
    return table[np.asarray(codes, np.uint8)] * scales.astype(np.float64)[..., None]


def gather_sequence_fp8(codes, scales, block_table, b, seq_len, kv_head):
    """Dequantised logical [L][D] float64 rows of one sequence and KV head."""
    S = codes.shape[2]
    t = np.arange(seq_len)
    phys = block_table[b, t // S].astype(np.int64)
    return dequantize_rows_e4m3(codes[phys, kv_head, t % S, :], scales[phys, kv_head, t % S])


def kv_append_fp8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, block_table, seq_lens):
    """Quantise the new token's K and V rows and write codes and scales at
    logical position L_b - 1.  Returns new pools; the inputs are untouched."""
    kc, vc = k_codes.copy(), v_codes.copy()
    ks, vs = k_scales.copy(), v_scales.copy()
    S = k_codes.shape[2]
    new_kc, new_ks = quantize_rows_e4m3(k_new)   # [B][Hkv][D], [B][Hkv]
    new_vc, new_vs = quantize_rows_e4m3(v_new)
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


def decode_attention_fp8(q, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens, scale,
                         heads=None):
    """Decode attention over the dequantised E4M3 cache, float64 [B][Hq][D].

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
            K = gather_sequence_fp8(k_codes, k_scales, block_table, b, L, g)
            V = gather_sequence_fp8(v_codes, v_scales, block_table, b, L, g)
            for h in hs:
                out[b, h] = attend_one(q[b, h], K, V, scale)
    return out
