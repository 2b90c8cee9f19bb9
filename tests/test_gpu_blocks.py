"""GPU checks of pa_copy_blocks (KV swap in/out and copies within a pool)
against the oracle's byte copy, and a swap round trip that decode must not
notice.  Pools live on the device or in pinned host memory.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from paged_kv_decode_24_gb300 import binding, workloads
from paged_kv_decode_24_gb300.runner import DeviceDecode
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


def _pairs(rng, n_src, n_dst, n):
    src = rng.integers(0, n_src, n)
    dst = rng.permutation(n_dst)[:n]          # distinct destinations
    return np.stack([src, dst], 1).astype(np.int32)


@pytest.mark.parametrize("where", ["d2d", "h2d", "d2h"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.int8, torch.float32])
def test_copy_blocks_bit_exact(where, dtype):
    rng = np.random.default_rng(71)
    block = {torch.float16: (8, 16, 128), torch.int8: (8, 16, 64), torch.float32: (8, 16)}[dtype]
    src_np = rng.integers(-100, 100, (37,) + block).astype(np.float32)
    dst_np = rng.integers(-100, 100, (29,) + block).astype(np.float32)
    src = torch.from_numpy(src_np).to(dtype)
    dst = torch.from_numpy(dst_np).to(dtype)
    src = src.cuda() if where in ("d2d", "d2h") else src.pin_memory()
    dst = dst.cuda() if where in ("d2d", "h2d") else dst.pin_memory()
    pairs_np = _pairs(rng, 37, 29, 20)
    pairs_np[3] = (40, pairs_np[3, 1])        # source out of range: skipped and flagged
    pairs = torch.from_numpy(pairs_np).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = oracle.copy_blocks(dst.cpu().numpy(), src.cpu().numpy(), pairs_np)
    binding.copy_blocks(dst, src, pairs, status)
    torch.cuda.synchronize()
    assert int(status.item()) == binding.PA_DEV_BAD_PAGE
    got = dst.cpu().numpy()
    assert np.array_equal(got.view(np.uint8), np.ascontiguousarray(want).view(np.uint8))


def test_copy_blocks_large_block_and_many_pairs():
    """Blocks bigger than one pass of the CTA, and more pairs than CTAs."""
    rng = np.random.default_rng(72)
    src = torch.from_numpy(rng.integers(-9, 9, (3000, 8, 16, 128)).astype(np.float16)).cuda()
    dst = torch.zeros((2600, 8, 16, 128), dtype=torch.float16, device="cuda")
    pairs_np = _pairs(rng, 3000, 2600, 2500)
    pairs = torch.from_numpy(pairs_np).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.copy_blocks(dst, src, pairs, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    idx_s = torch.from_numpy(pairs_np[:, 0].astype(np.int64)).cuda()
    idx_d = torch.from_numpy(pairs_np[:, 1].astype(np.int64)).cuda()
    assert torch.equal(dst[idx_d], src[idx_s])


def test_swap_round_trip_is_invisible_to_decode():
    """Allocate pages with the free list, swap two sequences out to pinned
    host memory, let other pages take their place, swap them back into fresh
    pages and rewrite their block-table rows: decode matches the oracle on
    the original cache."""
    w = workloads.make_custom(seq_lens=[40, 100, 17, 64], num_q_heads=8, num_kv_heads=2,
                              head_dim=128, num_pages=24, seed=73)
    want_dd = DeviceDecode(w)
    want_dd.make_plan()
    ref = want_dd.decode().cpu().numpy()

    dd = DeviceDecode(w)
    a = binding.BlockAllocator(w.num_pages)
    used = sorted(set(int(x) for x in w.block_table.ravel() if x >= 0))
    got = a.alloc(w.num_pages)             # the workload owns its pages; take them all
    a.free([p for p in got.tolist() if p not in used])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    host_k = torch.empty((w.num_pages,) + tuple(dd.k_pages.shape[1:]), dtype=torch.float16).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    bt = w.block_table.copy()
    for b in (1, 3):                        # swap out
        n = -(-int(w.seq_lens[b]) // 16)
        pages = bt[b, :n].copy()
        pairs = torch.from_numpy(np.stack([pages, np.arange(n) + 12 * (b // 2)], 1)
                                 .astype(np.int32)).cuda()
        binding.copy_blocks(host_k, dd.k_pages, pairs, status)
        binding.copy_blocks(host_v, dd.v_pages, pairs, status)
        torch.cuda.synchronize()
        a.free(pages)
        dd.k_pages[torch.from_numpy(pages.astype(np.int64)).cuda()] = 7.0   # reused by others
    for b in (3, 1):                        # swap in, into fresh pages
        n = -(-int(w.seq_lens[b]) // 16)
        fresh = a.alloc(n)
        pairs = torch.from_numpy(np.stack([np.arange(n) + 12 * (b // 2), fresh], 1)
                                 .astype(np.int32)).cuda()
        binding.copy_blocks(dd.k_pages, host_k, pairs, status)
        binding.copy_blocks(dd.v_pages, host_v, pairs, status)
        bt[b, :n] = fresh
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    dd.block_table.copy_(torch.from_numpy(bt))
    dd.make_plan()
    out = dd.decode().cpu().numpy()
    assert dd.read_status() == 0
    assert np.array_equal(out.view(np.uint16), ref.view(np.uint16))
    assert_close(out, oracle.decode_attention(w.q, w.k_pages, w.v_pages, w.block_table,
                                              w.seq_lens, w.scale), "after swap")
