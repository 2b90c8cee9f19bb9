"""Float64 CPU oracle (test infrastructure only; the library never imports it)."""

from .attention import (attend_one, decode_attention, decode_attention_split, gather_sequence,
                        gather_slots, kv_append, merge_partials, round_fp16, split_partial)

__all__ = ["attend_one", "decode_attention", "decode_attention_split", "gather_sequence",
           "gather_slots", "kv_append", "merge_partials", "round_fp16", "split_partial"]
