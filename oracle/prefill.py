"""Oracle for attention of several new query tokens per sequence over the
paged KV cache (chunked prefill, or prefill and decode tokens in one batch).

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module; the library never does, and this module
imports nothing from the library.

What it computes, and where the pages define it:

* "Eine LLM-Inferenz-Engine von Grund auf mit C++ und CUDA bauen",
  section 1.1: the prefill phase pushes the prompt tokens through the model
  and fills the KV cache; section 4 names processing several prompt tokens
  at once, and FlashAttention-style fused attention, as the next steps.
* swiftLLM, feature list: piggybacked prefill and decode (SARATHI) and
  Flash Attention, over PagedAttention's block tables.
* Each query token attends, like the decode token, with
  softmax(scale * K q) V, over the cached tokens up to its own position.

Readings of what the pages leave open:

* Sequence b has seq_lens[b] = L_b cached tokens, the newest q_lens[b] of
  which are this step's query tokens: query i sits at position
  L_b - q_lens[b] + i and attends positions 0 .. that position (causal).
  q_lens[b] <= L_b.  A decode token is the case q_lens[b] = 1.
* q, the new K/V rows and out are packed token-major, sequence after
  sequence: row cu[b] + i, cu = prefix sums of q_lens.
* The new rows are written into the pages first (token i at its position),
  as in the decode step.
"""

from __future__ import annotations

import numpy as np

from .attention import attend_one, gather_sequence


def cu_lens(q_lens) -> np.ndarray:
    """Prefix sums [B+1] of q_lens: sequence b's rows are cu[b] .. cu[b+1]-1."""
    return np.concatenate([[0], np.cumsum(np.asarray(q_lens, np.int64))])


def kv_append_tokens(k_pages, v_pages, k_new, v_new, block_table, seq_lens, q_lens):
    """Write the q_lens[b] new rows of every sequence at positions
    L_b - q_lens[b] .. L_b - 1.  Returns new pools; inputs are untouched."""
    k_out, v_out = k_pages.copy(), v_pages.copy()
    S = k_pages.shape[2]
    cu = cu_lens(q_lens)
    for b in range(len(seq_lens)):
        L, n = int(seq_lens[b]), int(q_lens[b])
        for i in range(n):
            pos = L - n + i
            page = int(block_table[b, pos // S])
            k_out[page, :, pos % S, :] = k_new[cu[b] + i]
            v_out[page, :, pos % S, :] = v_new[cu[b] + i]
    return k_out, v_out


def prefill_attention(q, k_pages, v_pages, block_table, seq_lens, q_lens, scale, rows=None):
    """Float64 out [T][Hq][D].  ``rows``, if given, lists the (row, head)
    pairs to compute; the others stay NaN."""
    T, Hq, D = q.shape
    Hkv = k_pages.shape[1]
    G = Hq // Hkv
    out = np.full((T, Hq, D), np.nan, np.float64)
    wanted = None if rows is None else set((int(r), int(h)) for r, h in rows)
    cu = cu_lens(q_lens)
    for b in range(len(seq_lens)):
        L, n = int(seq_lens[b]), int(q_lens[b])
        for g in range(Hkv):
            K = V = None
            for i in range(n):
                r = int(cu[b]) + i
                hs = [h for h in range(g * G, (g + 1) * G) if wanted is None or (r, h) in wanted]
                if not hs:
                    continue
                if K is None:
                    K = gather_sequence(k_pages, block_table, b, L, g)
                    V = gather_sequence(v_pages, block_table, b, L, g)
                p = L - n + i
                for h in hs:
                    out[r, h] = attend_one(q[r, h], K[:p + 1], V[:p + 1], scale)
    return out
