"""Float64 CPU oracle for decode attention over a paged KV cache.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module; the library never does, and this module
imports nothing from the library.  It is deliberately plain and slow.

What it computes, and where the pages define it:

* KV cache and the decode phase -- "Eine LLM-Inferenz-Engine von Grund auf
  mit C++ und CUDA bauen", section 1.1: prefill fills the KV cache, decode then
  produces one token at a time and attends over the cached keys and values.
* Paged KV cache (PagedAttention) -- swiftLLM, feature list: a sequence's
  cache lives in fixed-size pages found through a per-sequence block table.
* GQA -- MonadKai/xLLM, introduction (KV cache: GQA): several query heads
  share one KV head.
* The attended result softmax(q K^T * scale) V -- the plain definition of
  scaled dot-product attention for one query token.
* Flash-Decoding (paged attention v2) -- swiftLLM, feature list: the sequence
  is cut into chunks whose partial results are merged by a log-sum-exp
  combine.  ``decode_attention_split`` below writes that merge out only so the
  tests can show that any page-aligned split gives the unsplit answer.

Readings of what the pages leave open:

* GQA mapping: query head h reads KV head h // G, G = Hq / Hkv (consecutive
  query heads share a KV head).
* Logical token t of sequence b lives in physical page block_table[b][t // S],
  slot t % S; the pool is laid out [page][kv_head][slot][dim].
* seq_lens count the token being decoded; there is no other mask.
* A sequence of length 0 yields an all-zero output.
* fp16 inputs are widened exactly to float64; every operation is float64.
"""

from __future__ import annotations

import numpy as np


def gather_slots(block_table: np.ndarray, seq_lens: np.ndarray, page_size: int) -> np.ndarray:
    """Physical slot page * S + t % S of every logical token, -1 past the end.

    Output shape [B][max_pages * S]; the mapping is the paged-cache lookup of
    the swiftLLM feature list (PagedAttention).
    """
    B, max_pages = block_table.shape
    out = np.full((B, max_pages * page_size), -1, np.int64)
    for b in range(B):
        for t in range(int(seq_lens[b])):
            out[b, t] = int(block_table[b, t // page_size]) * page_size + t % page_size
    return out


def gather_sequence(pages: np.ndarray, block_table: np.ndarray, b: int, seq_len: int,
                    kv_head: int) -> np.ndarray:
    """Logical [L][D] float64 rows of one sequence and KV head, through the block table."""
    S = pages.shape[2]
    t = np.arange(seq_len)
    phys = block_table[b, t // S].astype(np.int64)
    return pages[phys, kv_head, t % S, :].astype(np.float64)


def kv_append(k_pages, v_pages, k_new, v_new, block_table, seq_lens):
    """Write the new token's K and V at logical position L_b - 1 (decode-phase
    cache update, section 1.1 of the from-scratch engine article).  Returns
    new pools; the inputs are left untouched.  Values are copied bit for bit."""
    k_out = k_pages.copy()
    v_out = v_pages.copy()
    S = k_pages.shape[2]
    for b in range(len(seq_lens)):
        pos = int(seq_lens[b]) - 1
        if pos < 0:
            continue
        page = int(block_table[b, pos // S])
        k_out[page, :, pos % S, :] = k_new[b]
        v_out[page, :, pos % S, :] = v_new[b]
    return k_out, v_out


def attend_one(q_row: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * keys @ q) @ values in float64 for one query vector."""
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1], np.float64)
    s = scale * (keys @ q_row.astype(np.float64))
    e = np.exp(s - s.max())
    p = e / e.sum()
    return p @ values


def decode_attention(q, k_pages, v_pages, block_table, seq_lens, scale, heads=None):
    """Decode attention for every (sequence, query head), float64 [B][Hq][D].

    ``heads``, if given, is an iterable of (b, h) pairs; only those outputs are
    computed (the others stay NaN) so large workloads can be sampled.
    """
    B, Hq, D = q.shape
    Hkv = k_pages.shape[1]
    G = Hq // Hkv
    out = np.full((B, Hq, D), np.nan, np.float64)
    wanted = None if heads is None else set((int(b), int(h)) for b, h in heads)
    for b in range(B):
        L = int(seq_lens[b])
        for g in range(Hkv):
            hs = [h for h in range(g * G, (g + 1) * G) if wanted is None or (b, h) in wanted]
            if not hs:
                continue
            K = gather_sequence(k_pages, block_table, b, L, g)
            V = gather_sequence(v_pages, block_table, b, L, g)
            for h in hs:
                out[b, h] = attend_one(q[b, h], K, V, scale)
    return out


def split_partial(q_row, keys, values, scale):
    """One Flash-Decoding chunk: its normalised output o and log-sum-exp of its scores."""
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1]), -np.inf
    s = scale * (keys @ q_row.astype(np.float64))
    m = s.max()
    e = np.exp(s - m)
    return (e @ values) / e.sum(), m + np.log(e.sum())


def merge_partials(partials):
    """Log-sum-exp merge of chunk results: out = sum_s exp(lse_s - LSE) o_s."""
    lses = np.array([lse for _, lse in partials])
    if np.all(np.isneginf(lses)):
        return np.zeros_like(partials[0][0])
    top = lses.max()
    lse_all = top + np.log(np.exp(lses - top).sum())
    return sum(np.exp(lse - lse_all) * o for o, lse in partials)


def decode_attention_split(q, k_pages, v_pages, block_table, seq_lens, scale, chunk_pages):
    """Flash-Decoding form of ``decode_attention``: each sequence is cut into
    page-aligned chunks of ``chunk_pages`` pages, each chunk yields (o, lse)
    and the chunks are merged with the log-sum-exp formula."""
    B, Hq, D = q.shape
    Hkv = k_pages.shape[1]
    S = k_pages.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), np.float64)
    step = chunk_pages * S
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(Hq):
            K = gather_sequence(k_pages, block_table, b, L, h // G)
            V = gather_sequence(v_pages, block_table, b, L, h // G)
            parts = [split_partial(q[b, h], K[t0:t0 + step], V[t0:t0 + step], scale)
                     for t0 in range(0, max(L, 1), step)]
            out[b, h] = merge_partials(parts)
    return out


def round_fp16(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even to fp16 (the output type), back to float64."""
    return x.astype(np.float16).astype(np.float64)
