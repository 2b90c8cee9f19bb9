"""Byte and FLOP accounting for the decode step (roofline numerators).

Decode attention reads every cached key and value once, so it is bound by HBM
bandwidth, not arithmetic: the roofline table of MonadKai/xLLM (section
"性能瓶颈分析") rates attention score and attention output at one FLOP per
byte for MHA.  The numbers below are the bytes the algorithm has to move,
independent of how a kernel moves them; split partials are kernel overhead
and are not counted.
"""

from __future__ import annotations

import numpy as np


def kv_cache_bytes(seq_lens, kv_width: int, bytes_per_element: int, layers: int = 1,
                   round_to: int = 1) -> int:
    """Bytes of a KV cache holding K and V for every token of every sequence.

    ``kv_width`` is Hkv * D (h1 for MHA).  Each sequence length is first rounded
    up to a multiple of ``round_to`` (the xLLM memory table rounds to 128).
    """
    lens = np.asarray(seq_lens, np.int64)
    rounded = (lens + round_to - 1) // round_to * round_to
    return int(2 * rounded.sum() * kv_width * bytes_per_element * layers)


def kv_row_bytes(head_dim: int, kv: str = "fp16") -> int:
    """Bytes of one cached row (one token, one KV head, K or V): D fp16 values,
    or D 8-bit codes and one fp32 scale (per-row INT8 or FP8 cache)."""
    if kv == "fp16":
        return 2 * head_dim
    if kv in ("int8", "fp8"):
        return head_dim + 4
    raise ValueError(kv)


def decode_bytes(seq_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 page_size: int, kv: str = "fp16") -> int:
    """Algorithmic HBM bytes of one decode-attention call (fp16 q/out).

    K and V of every attended token (fp16, INT8 or FP8 rows), q and out, the
    block-table entries that are read (one int32 per used page) and seq_lens.
    """
    lens = np.asarray(seq_lens, np.int64)
    B = len(lens)
    kv = int(2 * lens.sum() * num_kv_heads * kv_row_bytes(head_dim, kv))
    q_out = 2 * B * num_q_heads * head_dim * 2
    pages = int(((lens + page_size - 1) // page_size).sum())
    return int(kv + q_out + 4 * pages + 4 * B)


def append_bytes(batch: int, num_kv_heads: int, head_dim: int, kv: str = "fp16") -> int:
    """The append reads k_new, v_new (fp16) and writes one row of each."""
    rows = 2 * batch * num_kv_heads
    return rows * (2 * head_dim + kv_row_bytes(head_dim, kv))


def decode_flops(seq_lens, num_q_heads: int, head_dim: int) -> int:
    """2 FLOPs per multiply-add: q.k and p.v, D each, per token and query head."""
    return int(4 * head_dim * num_q_heads * np.asarray(seq_lens, np.int64).sum())
