"""The float64 oracle of an 8-bit cache workload (INT8 codes or FP8 bytes,
``w.kv``): its append, then decode attention over the new pools."""

from __future__ import annotations

import oracle


def oracle_append_decode(w, heads=None):
    """(out float64 [B][Hq][D], (k_codes, v_codes, k_scales, v_scales)) after the append."""
    append, decode = ((oracle.kv_append_fp8, oracle.decode_attention_fp8) if w.kv == "fp8" else
                      (oracle.kv_append_q8, oracle.decode_attention_q8))
    kc, vc, ks, vs = append(w.k_codes, w.v_codes, w.k_scales, w.v_scales, w.k_new, w.v_new,
                            w.block_table, w.seq_lens)
    out = decode(w.q, kc, vc, ks, vs, w.block_table, w.seq_lens, w.scale, heads=heads)
    return out, (kc, vc, ks, vs)


def oracle_decode(w, heads=None):
    """Decode attention over the workload's 8-bit pools as they are (no append)."""
    decode = oracle.decode_attention_fp8 if w.kv == "fp8" else oracle.decode_attention_q8
    return decode(w.q, w.k_codes, w.v_codes, w.k_scales, w.v_scales, w.block_table, w.seq_lens,
                  w.scale, heads=heads)
