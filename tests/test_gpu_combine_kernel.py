"""The two-kernel form of the split merge: a plan made with
merge = PA_MERGE_COMBINE_KERNEL has its split tasks only write partials, and a
separate combine kernel, launched after the split kernel, merges them (the
Flash-Decoding reduce as its own launch).  The form is chosen per plan, so
both forms run here in one process, on the same inputs.  Outputs must match
the oracle for each split kernel (CUDA cores, tensor cores, INT8 cache) and
element type, agree with the default in-kernel merge to rounding, give the
same bits on every call, and leave the workspace's group counters at zero.
"""

from __future__ import annotations

import zlib

import numpy as np
import pytest

import oracle
from paged_kv_decode_24_gb300 import workloads
from paged_kv_decode_24_gb300.runner import DeviceDecode
from tests.cache8 import oracle_append_decode
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


def counters(dd):
    blob = dd.plan_obj.blob()
    W, C = int(blob[1]), int(blob[2])
    c0 = (16 + 6 * W + 3) // 4 * 4 + 4 * C
    return dd.workspace[:(c0 + C) * 4].view(torch.int32)[c0:c0 + C].cpu().numpy()


def oracle_step(w):
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    return oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)


CASES = [([5, 300, 129, 1000], 32, 8, 128, 0, "fp16"), ([96, 97, 1500], 16, 16, 128, 7, "fp16"),
         ([2000, 3, 640], 4, 4, 64, 0, "fp16"), ([1500, 700, 33], 16, 4, 128, 5, "bf16"),
         ([4096], 32, 32, 128, 16, "fp16")]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"L{c[0][:2]}_G{c[1] // c[2]}_D{c[3]}_{c[5]}")
def test_two_kernel_form_matches_oracle(case):
    lens, hq, hkv, d, splits, dtype = case
    w = workloads.make_custom(seq_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              seed=zlib.crc32(str(case).encode()) ^ 11, forced_splits=splits,
                              dtype=dtype)
    dd = DeviceDecode(w)
    dd.append()
    want = oracle_step(w)
    outs = {}
    for merge in ("combine", "split", "combine"):   # both forms, alternating, one process
        dd.make_plan(forced_splits=splits, merge=merge)
        assert dd.plan_obj.c.num_groups > 0
        first = dd.decode().clone()
        assert dd.read_status() == 0, dd.read_status()
        assert_close(first.float().cpu().numpy(), want, f"{merge} merge {case}", dtype=dtype)
        for _ in range(5):
            assert torch.equal(dd.decode().view(torch.int16), first.view(torch.int16))
        assert np.all(counters(dd) == 0)
        if merge in outs:   # each form gives the same bits whenever it runs
            assert torch.equal(outs[merge].view(torch.int16), first.view(torch.int16))
        outs[merge] = first


@pytest.mark.parametrize("kv", ["int8", "fp8"])
def test_two_kernel_form_8bit_cache(kv):
    w = workloads.make_custom(seq_lens=[700, 33, 1024], num_q_heads=32, num_kv_heads=8,
                              head_dim=128, seed=83, kv=kv, forced_splits=4)
    dd = DeviceDecode(w)
    dd.make_plan(merge="combine")
    dd.append8()
    got = dd.decode8().cpu().numpy()
    assert dd.read_status() == 0
    want, _ = oracle_append_decode(w)
    assert_close(got, want, f"combine kernel, {kv} cache")
