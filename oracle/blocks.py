"""Oracle for KV block management: page counts, the free list, block copies.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module; the library never does, and this module
imports nothing from the library.

What it computes, and where the pages define it:

* swiftLLM, architecture section: the engine has its worker profile the
  number of GPU blocks, then allocates the KV cache and a KV swap space, and
  every step swaps blocks in and out before the compute.
* MonadKai/xLLM, memory table: the KV cache holds 2 (K and V) x b x h1 x L
  elements per token position, the size a page count is derived from.

Readings of what the pages leave open:

* A block is one page: page_size tokens of every KV head of one layer's K
  (or V) pool.  Pages needed for num_layers layers' K and V:
  2 x Hkv x page_size x row_bytes x num_layers bytes each, row_bytes =
  2 x head_dim for 16-bit elements, head_dim + 4 for 8-bit codes (INT8 or
  FP8) plus an fp32 scale.  The page count is floor((free - reserve) / that).
* The free list hands pages out last-freed first; a fresh list hands out
  0, 1, 2, ...  Allocation is all or nothing; freeing a page that is not
  out, out of range, or listed twice is refused and frees nothing.
* A block copy is a byte copy of whole blocks, dst[d] = src[s] per pair.
"""

from __future__ import annotations

import numpy as np


def row_bytes(head_dim: int, kind: str) -> int:
    return 2 * head_dim if kind == "16bit" else head_dim + 4


def profile_num_blocks(num_kv_heads, page_size, head_dim, num_layers, kind, free_bytes,
                       reserve_bytes):
    if free_bytes <= reserve_bytes:
        return 0
    per_page = 2 * num_kv_heads * page_size * row_bytes(head_dim, kind) * num_layers
    return (free_bytes - reserve_bytes) // per_page


class BlockAllocatorModel:
    """The free list, written plainly: a Python list used as a stack."""

    def __init__(self, num_blocks: int):
        self.stack = list(range(num_blocks - 1, -1, -1))
        self.out = set()
        self.n = num_blocks

    def num_free(self) -> int:
        return len(self.stack)

    def alloc(self, k: int):
        """k pages, or None (and nothing taken) when fewer are free."""
        if k > len(self.stack):
            return None
        got = [self.stack.pop() for _ in range(k)]
        self.out.update(got)
        return got

    def free(self, blocks) -> bool:
        """True if freed; False (nothing freed) for a bad list."""
        blocks = list(blocks)
        if len(set(blocks)) != len(blocks) or any(b not in self.out for b in blocks):
            return False
        for b in blocks:
            self.out.remove(b)
            self.stack.append(b)
        return True

    def grow(self, row, page_size, old_len, new_len):
        """Fill row entries [ceil(old/S), ceil(new/S)) with fresh pages; False
        (row untouched) when the pool is short."""
        have = -(-old_len // page_size)
        need = -(-new_len // page_size)
        got = self.alloc(need - have)
        if got is None:
            return False
        row[have:need] = got
        return True


def copy_blocks(dst: np.ndarray, src: np.ndarray, pairs) -> np.ndarray:
    """dst with block d replaced by block s of src for every (s, d) pair; a
    pair out of range is skipped.  Blocks are the first axis."""
    out = dst.copy()
    for s, d in np.asarray(pairs).reshape(-1, 2):
        if 0 <= s < src.shape[0] and 0 <= d < dst.shape[0]:
            out[d] = src[s]
    return out
