"""KV block management without a GPU: the oracle's pins, and the library's
page count and free list against the oracle.

Pins: the page count reproduces the xLLM memory table (30 GiB of fp32 cache
for its batch is 15 GiB, 1920 pages, of fp16); the block copy equals an
element-by-element loop; the free-list model keeps its invariants under a
seeded random walk.  The library's allocator then follows the same walk and
must hand out exactly the model's pages and refuse exactly what it refuses.
"""

from __future__ import annotations

import os

import numpy as np
import pytest

import oracle
from paged_kv_decode_24_gb300 import binding

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_memory.txt")


def _golden():
    vals = {}
    for raw in open(GOLDEN):
        line = raw.split("#", 1)[0].strip()
        if line:
            k, v = (x.strip() for x in line.split("="))
            vals[k] = int(v)
    return vals


def test_oracle_page_count_matches_xllm_table():
    g = _golden()
    tokens = g["b"] * (-(-(g["s"] + g["n"]) // g["round_to"]) * g["round_to"])
    # the table's cache is fp32 (4 bytes); the same tokens in 16-bit elements take half
    fp16_bytes = g["expect_gib"] * 2**30 * 2 // g["bytes_per_element"]
    pages = oracle.profile_num_blocks(32, 16, 128, g["layers"], "16bit", fp16_bytes, 0)
    assert 32 * 128 == g["h1"]
    assert pages * 16 == tokens == 30720
    assert oracle.profile_num_blocks(32, 16, 128, 32, "16bit", fp16_bytes - 1, 0) == pages - 1
    assert oracle.profile_num_blocks(32, 16, 128, 32, "16bit", 100, 200) == 0


def test_oracle_copy_blocks_is_an_elementwise_copy():
    rng = np.random.default_rng(61)
    src = rng.standard_normal((7, 2, 3))
    dst = rng.standard_normal((5, 2, 3))
    pairs = [(6, 0), (0, 4), (3, 2), (9, 1)]      # the last is out of range: skipped
    got = oracle.copy_blocks(dst, src, pairs)
    want = dst.copy()
    for s, d in pairs:
        if s < 7 and d < 5:
            for i in range(2):
                for j in range(3):
                    want[d, i, j] = src[s, i, j]
    assert np.array_equal(got, want)
    assert np.array_equal(got[[1, 3]], dst[[1, 3]])


def _walk(seed, n_blocks, steps):
    """A seeded mix of allocs, frees (some invalid) and grows."""
    rng = np.random.default_rng(seed)
    ops = []
    for _ in range(steps):
        r = rng.random()
        if r < 0.45:
            ops.append(("alloc", int(rng.integers(0, n_blocks // 3 + 2))))
        elif r < 0.85:
            ops.append(("free", None))
        else:
            ops.append(("bad_free", int(rng.integers(-2, n_blocks + 2))))
    return ops


def test_oracle_allocator_invariants():
    m = oracle.BlockAllocatorModel(40)
    assert m.alloc(3) == [0, 1, 2]
    assert m.free([1]) and m.alloc(1) == [1]           # last freed, first out
    assert m.alloc(38) is None and m.num_free() == 37  # all or nothing
    assert not m.free([1, 1]) and not m.free([39]) and m.num_free() == 37
    row = np.full(8, -1, np.int32)
    assert m.grow(row, 16, 0, 33) and list(row[:3]) == [3, 4, 5] and row[3] == -1
    assert m.grow(row, 16, 33, 48) and row[3] == -1    # still 3 pages
    assert m.grow(row, 16, 48, 49) and row[3] == 6


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_library_allocator_follows_the_model(lib, seed):
    n_blocks = 64
    a = binding.BlockAllocator(n_blocks)
    m = oracle.BlockAllocatorModel(n_blocks)
    rng = np.random.default_rng(seed + 100)
    held = []
    for op, arg in _walk(seed, n_blocks, 300):
        if op == "alloc":
            want = m.alloc(arg)
            if want is None:
                with pytest.raises(binding.PagedAttnError) as e:
                    a.alloc(arg)
                assert e.value.code == 7
            else:
                got = a.alloc(arg)
                assert got.tolist() == want
                held.extend(want)
        elif op == "free" and held:
            k = int(rng.integers(1, len(held) + 1))
            pick = [held.pop(int(rng.integers(0, len(held)))) for _ in range(k)]
            assert m.free(pick)
            a.free(pick)
        elif op == "bad_free":
            bad = [arg] + ([held[0], held[0]] if held and arg % 2 == 0 else [])
            if not m.free(bad):
                with pytest.raises(binding.PagedAttnError) as e:
                    a.free(bad)
                assert e.value.code == 1
            else:
                a.free(bad)
                held = [h for h in held if h not in bad]
        assert a.num_free() == m.num_free()
    a.close()


def test_library_grow_and_page_count(lib):
    a = binding.BlockAllocator(5)
    row = np.full(4, -1, np.int32)
    a.grow(row, 16, 0, 17)
    assert row.tolist() == [0, 1, -1, -1]
    a.grow(row, 16, 17, 32)
    assert row.tolist() == [0, 1, -1, -1]
    with pytest.raises(binding.PagedAttnError) as e:
        a.grow(row, 16, 32, 65)        # 5 pages > 4 entries
    assert e.value.code == 1
    a.grow(row, 16, 32, 64)
    assert row.tolist() == [0, 1, 2, 3] and a.num_free() == 1
    with pytest.raises(binding.PagedAttnError) as e:
        binding.BlockAllocator(1).grow(np.full(4, -1, np.int32), 16, 0, 40)   # pool short
    assert e.value.code == 7
    for kv, kind, d in ((binding.PA_KV_16BIT, "16bit", 128), (binding.PA_KV_INT8, "int8", 64),
                        (binding.PA_KV_FP8, "fp8", 128)):
        s = binding.make_shape(4, 32, 8, d, 16, 64, 100)
        for free, reserve in ((80 * 2**30, 2**30), (12345678, 0), (10, 20)):
            assert binding.profile_num_blocks(s, 32, kv, free, reserve) == \
                oracle.profile_num_blocks(8, 16, d, 32, kind, free, reserve)
