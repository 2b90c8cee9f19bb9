"""The L2 prefetch that the split-decode kernels issue before waiting on the
previous kernel, at its widest setting (plan options): every CTA and all 32
lanes of every warp prefetch, so every block-table entry a warp owns goes
through the bounds checks.  Results must match the oracle as with the
default setting, and a block-table entry outside the pool must be flagged and
skipped, not prefetched.  The setting with no prefetch at all must match too.
"""

from __future__ import annotations

import zlib

import numpy as np
import pytest

import oracle
from paged_kv_decode_24_gb300 import binding, workloads
from paged_kv_decode_24_gb300.runner import DeviceDecode
from tests.cache8 import oracle_append_decode
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

WIDEST = dict(l2_prefetch_pages=32, l2_prefetch_ctas=2147483647)
NONE = dict(l2_prefetch_pages=-1, l2_prefetch_ctas=-1)


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


def oracle_step(w):
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    return oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)


@pytest.mark.parametrize("opts", [WIDEST, NONE], ids=["widest", "none"])
@pytest.mark.parametrize("case", [([5, 300, 129, 1000], 32, 8, 128, 0),
                                  ([96, 97, 1500], 16, 16, 128, 7), ([2000, 3, 640], 4, 4, 64, 0)],
                         ids=lambda c: f"L{c[0][:2]}_G{c[1] // c[2]}_D{c[3]}")
def test_prefetch_setting_matches_oracle(case, opts):
    lens, hq, hkv, d, splits = case
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              seed=zlib.crc32(str(case).encode()) ^ 7, forced_splits=splits)
    dd = DeviceDecode(w)
    dd.append()
    dd.make_plan(forced_splits=splits, **opts)
    got = dd.decode().cpu().numpy()
    assert dd.read_status() == 0, dd.read_status()
    assert_close(got, oracle_step(w), f"prefetch {opts} {case}")


@pytest.mark.parametrize("kv", ["int8", "fp8"])
def test_widest_prefetch_8bit_cache(kv):
    w = workloads.make_custom(seq_lens=[700, 33, 1024], num_q_heads=32, num_kv_heads=8,
                              head_dim=128, seed=71, kv=kv)
    dd = DeviceDecode(w)
    dd.make_plan(**WIDEST)
    dd.append8()
    got = dd.decode8().cpu().numpy()
    assert dd.read_status() == 0
    want, _ = oracle_append_decode(w)
    assert_close(got, want, f"prefetch {kv}")


def test_widest_prefetch_skips_a_bad_entry():
    """An entry outside the pool: flagged, skipped, never prefetched."""
    w = workloads.make_custom(seq_lens=[40, 400], num_q_heads=4, num_kv_heads=2, head_dim=64,
                              seed=72)
    w.block_table[1, 3] = w.num_pages + 1000
    dd = DeviceDecode(w)
    dd.make_plan(**WIDEST)
    out = dd.decode().cpu().numpy()
    assert dd.read_status() & binding.PA_DEV_BAD_PAGE
    assert np.all(np.isfinite(out.astype(np.float32)))
