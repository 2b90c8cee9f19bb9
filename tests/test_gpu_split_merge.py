"""GPU: the split merge, run by the last split task of each group.

A split task adds one to its group's counter after writing its partial; the
task that completes the group merges the partials into out and sets the
counter back to zero.  Which task merges depends on timing.  These tests
check, against the float64 oracle and across repeated calls:
- a group whose split tasks mix the two task forms (a CTA's warps sharing a
  task, and a task run by one warp of a bundle) merges to the oracle's
  result and to the same bits on every call, for each split kernel;
- every counter is zero again after a call, and many calls on one upload
  agree bit for bit.
"""

from __future__ import annotations

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


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


def blob_parts(plan):
    """Tasks, their {slot, group} words, the counters' int32 offset and the
    number of CTA-shared tasks, from the plan's host copy."""
    blob = plan.blob()
    W, C = int(blob[1]), int(blob[2])
    items = blob[16:16 + 4 * W].reshape(W, 4)
    sg = blob[16 + 4 * W:16 + 6 * W].reshape(W, 2)
    g0 = (16 + 6 * W + 3) // 4 * 4
    return items, sg, g0 + 4 * C, C, int(blob[9])


def counters(dd):
    _, _, c0, C, _ = blob_parts(dd.plan_obj)
    return dd.workspace[:(c0 + C) * 4].view(torch.int32)[c0:c0 + C].cpu().numpy()


def mixed_groups(plan):
    """Groups with both a CTA-shared task and a per-warp task."""
    items, sg, _, _, n_shared = blob_parts(plan)
    kinds = {}
    for i in range(len(items)):
        if sg[i, 0] >= 0:
            kinds.setdefault(int(sg[i, 1]), set()).add(i < n_shared)
    return [g for g, k in kinds.items() if k == {True, False}]


def mixed_workload(num_q_heads, kv="fp16", dtype="fp16", seed=71):
    # 17-page sequences cut in two give 8- and 9-page splits.  Planned for one
    # SM (four CTA slots) the 32+ tasks are many, so the 8-page ones are
    # bundled one per warp while the 9-page ones get a CTA each.
    return workloads.make_custom(seq_lens=[272, 270, 260, 258, 50], num_q_heads=num_q_heads,
                                 num_kv_heads=4, head_dim=128, seed=seed, forced_splits=2,
                                 kv=kv, dtype=dtype)


@pytest.mark.parametrize("num_q_heads,dtype", [(4, "fp16"), (16, "fp16"), (16, "bf16")])
def test_mixed_task_forms_merge_to_oracle_and_same_bits(num_q_heads, dtype):
    w = mixed_workload(num_q_heads, dtype=dtype)
    dd = DeviceDecode(w, num_sms=1)
    dd.append()
    dd.make_plan()
    assert mixed_groups(dd.plan_obj), "the plan has no group that mixes the task forms"
    first = dd.decode().clone()
    assert dd.read_status() == 0
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
    assert_close(first.float().cpu().numpy(), want, "mixed task forms", dtype=dtype)
    assert np.all(counters(dd) == 0)
    for _ in range(20):
        again = dd.decode()
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))
    assert np.all(counters(dd) == 0)


@pytest.mark.parametrize("kv", ["int8", "fp8"])
@pytest.mark.parametrize("num_q_heads", [4, 16])
def test_mixed_task_forms_8bit_cache(num_q_heads, kv):
    w = mixed_workload(num_q_heads, kv=kv, seed=73)
    dd = DeviceDecode(w, num_sms=1)
    dd.append8()
    dd.make_plan()
    assert mixed_groups(dd.plan_obj)
    first = dd.decode8().clone()
    assert dd.read_status() == 0
    want, _ = oracle_append_decode(w)
    assert_close(first.cpu().numpy(), want, f"mixed task forms, {kv} cache")
    for _ in range(20):
        assert torch.equal(dd.decode8().view(torch.int16), first.view(torch.int16))
    assert np.all(counters(dd) == 0)


def test_many_calls_on_one_upload():
    """200 calls on one uploaded plan of the default workload's shape (one
    sequence, 32 heads, 16 splits): identical outputs, counters at zero."""
    w = workloads.make_custom(seq_lens=[4096], num_q_heads=32, num_kv_heads=32, head_dim=128,
                              seed=79, forced_splits=16)
    dd = DeviceDecode(w)
    dd.append()
    dd.make_plan()
    assert dd.plan_obj.c.num_groups == 32
    first = dd.decode().clone()
    outs = [dd.decode().clone() for _ in range(200)]
    torch.cuda.synchronize()
    assert dd.read_status() == 0
    assert all(torch.equal(o.view(torch.int16), first.view(torch.int16)) for o in outs)
    assert np.all(counters(dd) == 0)
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    heads = [(0, h) for h in (0, 7, 31)]
    want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale, heads=heads)
    got = first.cpu().numpy()
    for (b, h) in heads:
        assert_close(got[b, h], want[b, h], f"head {h}")


def test_corrupted_group_words_are_flagged_and_upload_recovers():
    """Split tasks check their {slot, group} word and the group record
    against their own task before touching a partial or a counter.  A
    workspace whose words are corrupted is flagged PA_DEV_PLAN_MISMATCH;
    uploading the plan again restores the task list and zeroes the counters,
    and the next call matches the oracle."""
    w = workloads.make_custom(seq_lens=[600, 300, 900], num_q_heads=8, num_kv_heads=2,
                              head_dim=128, seed=97, forced_splits=3)
    dd = DeviceDecode(w)
    dd.append()
    dd.make_plan()
    items, sg, c0, C, _ = blob_parts(dd.plan_obj)
    W = len(items)
    g0 = (16 + 6 * W + 3) // 4 * 4
    split = np.nonzero(sg[:, 0] >= 0)[0]
    assert len(split) > 3 and C > 1
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.seq_lens)
    want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)

    def corrupt(edit):
        words = dd.workspace[:(g0 + 4 * C) * 4].view(torch.int32)
        edit(words)
        dd.status.zero_()
        dd.decode()
        assert dd.read_status() & binding.PA_DEV_PLAN_MISMATCH
        dd.status.zero_()
        binding.upload(dd.plan_obj, dd.workspace)
        got = dd.decode().cpu().numpy()
        assert dd.read_status() == 0
        assert np.all(counters(dd) == 0)
        assert_close(got, want, "after a fresh upload")

    def every_split_task_to_group_0(words):
        for i in split:
            words[16 + 4 * W + 2 * int(i) + 1] = 0

    def group_1_split_count_zero(words):
        words[g0 + 4 * 1 + 2] = 0

    def group_index_out_of_range(words):
        words[16 + 4 * W + 2 * int(split[0]) + 1] = C + 5

    corrupt(every_split_task_to_group_0)
    corrupt(group_1_split_count_zero)
    corrupt(group_index_out_of_range)
