"""Float64 CPU oracle (test infrastructure only; the library never imports it)."""

from .attention import (attend_one, decode_attention, decode_attention_split, gather_sequence,
                        gather_slots, kv_append, merge_partials, round_fp16, split_partial)
from .blocks import BlockAllocatorModel, copy_blocks, profile_num_blocks
from .fp8 import (decode_attention_fp8, dequantize_rows_e4m3, e4m3_encode, e4m3_round, e4m3_value,
                  kv_append_fp8, quantize_rows_e4m3)
from .prefill import cu_lens, kv_append_tokens, prefill_attention
from .quant import (decode_attention_q8, dequantize_rows, gather_sequence_q8, kv_append_q8,
                    quantize_rows_int8)

__all__ = ["attend_one", "decode_attention", "decode_attention_split", "gather_sequence",
           "gather_slots", "kv_append", "merge_partials", "round_fp16", "split_partial",
           "decode_attention_q8", "dequantize_rows", "gather_sequence_q8", "kv_append_q8",
           "quantize_rows_int8", "BlockAllocatorModel", "copy_blocks", "profile_num_blocks",
           "cu_lens", "kv_append_tokens", "prefill_attention", "decode_attention_fp8",
           "dequantize_rows_e4m3", "e4m3_encode", "e4m3_round", "e4m3_value", "kv_append_fp8",
           "quantize_rows_e4m3"]
