"""Host-side checks of libpagedattn that need no GPU.

The library loads and exports every function include/pagedattn.h declares.
pa_plan is pure host code, so its task list can be checked in full here.
Argument errors are rejected before any CUDA call.
"""

from __future__ import annotations

import ctypes
import types

import numpy as np
import pytest

from paged_kv_decode_24_gb300 import binding, workloads


def test_exports_every_declared_symbol(lib):
    names = binding.declared_functions()
    assert {"pa_kv_append", "pa_plan", "pa_plan_free", "pa_plan_upload", "pa_decode_attention",
            "pa_debug_gather_indices", "pa_status_string", "pa_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in the header but not exported"


def test_status_strings(lib):
    for code in range(9):
        assert lib.pa_status_string(code)
    assert b"sm_103a" in lib.pa_version()


def _shape(w):
    return binding.make_shape(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size,
                              w.max_pages_per_seq, w.num_pages)


def _decode_blob(plan):
    """Header (16 int32) | tasks (4 int32 each) | task slots (2 int32 each:
    partial slot, group; padded to 16 bytes) | groups (4 int32 each) | group
    counters (1 int32 each, zero in the plan)."""
    blob = plan.blob()
    W, C, nslots = blob[1], blob[2], blob[3]
    items = blob[16:16 + 4 * W].reshape(W, 4)
    sg = blob[16 + 4 * W:16 + 6 * W].reshape(W, 2)
    slots, task_group = sg[:, 0], sg[:, 1]
    g0 = (16 + 6 * W + 3) // 4 * 4
    groups = blob[g0:g0 + 4 * C].reshape(C, 4)
    counters = blob[g0 + 4 * C:g0 + 5 * C]
    assert len(counters) == C and np.all(counters == 0)
    for i in range(W):  # a split task names the group of its own (sequence, head)
        if slots[i] >= 0:
            b, h = groups[task_group[i]][:2]
            assert (b, h) == (items[i][0], int(items[i][1]) & 0xFFFF)
        else:
            assert task_group[i] == -1
    NC, n_shared = blob[8], blob[9]
    return blob, items, groups, slots, nslots, (NC, n_shared)


def check_plan_covers(w, plan, bundle_max=8):
    """Every (sequence, kv head) has its pages [0, ceil(L/S)) covered exactly
    once by page ranges, split tasks appear in their group in page order, and
    tasks are longest first."""
    blob, items, groups, slots, nslots, ctas = _decode_blob(plan)
    assert blob[0] == 0x564B4150
    S = w.page_size
    cover = {}
    for i, (b, hw, lo, hi) in enumerate(items):
        hw = int(hw) & 0xFFFFFFFF
        h = hw & 0xFFFF
        cover.setdefault((int(b), h), []).append((int(lo), int(hi), i, bool(hw & 0x80000000),
                                                  bool(hw & 0x40000000)))
    assert len(cover) == w.batch * w.num_kv_heads
    for b in range(w.batch):
        npg = (int(w.seq_lens[b]) + S - 1) // S
        for h in range(w.num_kv_heads):
            ranges = sorted(cover[(b, h)])
            assert ranges[0][0] == 0 and ranges[-1][1] == npg
            for (lo0, hi0, *_), (lo1, *_r) in zip(ranges, ranges[1:]):
                assert hi0 == lo1
            split = len(ranges) > 1
            assert all(r[3] == split for r in ranges)
            assert [r[4] for r in ranges] == [False] * (len(ranges) - 1) + [True]
    sizes = items[:, 3] - items[:, 2]
    assert np.all(np.diff(sizes) <= 0), "tasks are not longest first"
    # split tasks own consecutive partial slots per group, in page order;
    # direct tasks own none
    seen = set()
    for (b, h, n, off) in groups:
        assert n > 1
        ranges = sorted(cover[(int(b), int(h))])
        assert [int(slots[r[2]]) for r in ranges] == list(range(off, off + n))
        seen.update(range(off, off + n))
    assert seen == set(range(nslots))
    for i, (b, hw, lo, hi) in enumerate(items):
        if not (int(hw) & 0x80000000):
            assert slots[i] == -1
    # CTAs: the first n_shared tasks get a CTA each; the remaining (short,
    # <= 8 pages) tasks go four to a CTA
    NC, n_shared = ctas
    assert plan.c.num_ctas == NC and plan.c.num_shared_ctas == n_shared
    assert 0 <= n_shared <= len(items)
    assert NC == n_shared + (len(items) - n_shared + 3) // 4
    assert np.all(sizes[n_shared:] <= bundle_max)
    assert plan.c.workspace_bytes >= plan.c.blob_bytes
    return items, groups


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_plan_for_benchmark_workloads(lib, cfg):
    w = workloads.make_config(cfg)
    plan = binding.Plan(_shape(w), w.seq_lens, 152, w.forced_splits)
    items, groups = check_plan_covers(w, plan)
    if cfg == 1:
        assert plan.c.num_groups == 0 and plan.c.num_work_items == w.batch * w.num_kv_heads
    if cfg == 2:
        assert plan.c.max_splits == 16 and plan.c.num_work_items == 16 * 32
        assert np.all(items[:, 3] - items[:, 2] == 16)
    if cfg == 5:
        # the 32k sequence is cut, the short ones are not
        assert plan.c.max_splits > 8
        long_items = items[items[:, 0] == 255]
        assert len(long_items) == plan.c.max_splits * w.num_kv_heads


@pytest.mark.parametrize("lens", [[0], [0, 0, 3], [1], [16], [17], [4095, 1, 0, 33]])
@pytest.mark.parametrize("forced", [0, 1, 3, 16])
def test_plan_ragged_and_empty(lib, lens, forced):
    w = workloads.make_custom(seq_lens=lens, num_q_heads=8, num_kv_heads=2, head_dim=128, seed=1)
    plan = binding.Plan(_shape(w), w.seq_lens, 152, forced)
    check_plan_covers(w, plan)


def test_plan_rejects_bad_inputs(lib):
    w = workloads.make_custom(seq_lens=[10, 20], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=2)
    s = _shape(w)
    with pytest.raises(binding.PagedAttnError) as e:
        binding.Plan(s, [10, w.max_pages_per_seq * 16 + 1], 152)
    assert e.value.code == 1
    with pytest.raises(binding.PagedAttnError) as e:
        binding.Plan(s, [-1, 5], 152)
    assert e.value.code == 1
    with pytest.raises(binding.PagedAttnError) as e:
        binding.Plan(s, [10, 20], 0)
    assert e.value.code == 1
    for bad, code in [(dict(head_dim=96), 2), (dict(page_size=8), 2), (dict(num_q_heads=6), 2),
                      (dict(num_q_heads=5), 1), (dict(num_kv_heads=0), 1), (dict(num_pages=0), 1)]:
        kw = dict(batch=2, num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16,
                  max_pages_per_seq=w.max_pages_per_seq, num_pages=w.num_pages)
        kw.update(bad)
        with pytest.raises(binding.PagedAttnError) as e:
            binding.Plan(binding.make_shape(**kw), [10, 20], 152)
        assert e.value.code == code, bad


def test_dtype_is_checked(lib):
    """fp16 and bf16 plan; any other dtype is unsupported; the INT8-cache calls
    take fp16 only (all refused before any CUDA call)."""
    kw = dict(batch=2, num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16,
              max_pages_per_seq=4, num_pages=8)
    for dt in ("fp16", "bf16"):
        binding.Plan(binding.make_shape(**kw, dtype=dt), [10, 20], 152)
    with pytest.raises(binding.PagedAttnError) as e:
        binding.Plan(binding.make_shape(**kw, dtype=2), [10, 20], 152)
    assert e.value.code == 2
    s = binding.make_shape(**kw, dtype="bf16")
    plan = binding.Plan(s, [10, 20], 152)
    fake = ctypes.c_void_p(0x10000)
    assert lib.pa_kv_append_q8(ctypes.byref(s), fake, fake, fake, fake, fake, fake, fake, fake,
                               fake, None) == 2
    assert lib.pa_decode_attention_q8(ctypes.byref(s), ctypes.byref(plan.c), fake, fake, fake,
                                      fake, fake, fake, fake, ctypes.c_float(0.1), fake, fake,
                                      plan.c.workspace_bytes, fake, None) == 2


def test_plan_free_is_idempotent(lib):
    w = workloads.make_custom(seq_lens=[5], num_q_heads=1, num_kv_heads=1, head_dim=64, seed=3)
    plan = binding.Plan(_shape(w), w.seq_lens, 152)
    plan.free()
    plan.free()
    lib.pa_plan_free(None)


def test_plan_is_deterministic_but_ids_differ(lib):
    w = workloads.make_config(4)
    a = binding.Plan(_shape(w), w.seq_lens, 152)
    b = binding.Plan(_shape(w), w.seq_lens, 152)
    ba, bb = a.blob(), b.blob()
    assert np.array_equal(np.delete(ba, [4, 5]), np.delete(bb, [4, 5]))
    assert a.c.plan_id != b.c.plan_id


def test_plan_in_caller_buffer(lib):
    w = workloads.make_config(3)
    s = _shape(w)
    ref = binding.Plan(s, w.seq_lens, 152)
    small = np.zeros(16, np.uint8)
    with pytest.raises(binding.PagedAttnError) as e:
        binding.Plan(s, w.seq_lens, 152, host_buffer=small)
    assert e.value.code == 3
    # a dirty buffer: every byte of the plan, gaps and group counters
    # included, is written (the kernels need the counters at zero)
    buf = np.full(ref.c.blob_bytes + 64, 0xFF, np.uint8)
    p = binding.Plan(s, w.seq_lens, 152, host_buffer=buf)
    assert p.c.owns_blob == 0 and p.c.host_blob == buf.ctypes.data
    got = buf[:ref.c.blob_bytes].view(np.int32)
    assert np.array_equal(np.delete(got, [4, 5]), np.delete(ref.blob(), [4, 5]))
    # the same with split groups, whose counters must come out zero
    w2 = workloads.make_custom(seq_lens=[3000, 50, 700], num_q_heads=8, num_kv_heads=2,
                               head_dim=128, seed=5)
    s2 = _shape(w2)
    ref2 = binding.Plan(s2, w2.seq_lens, 152, 4)
    buf2 = np.full(ref2.c.blob_bytes, 0xFF, np.uint8)
    binding.Plan(s2, w2.seq_lens, 152, 4, host_buffer=buf2)
    got2 = buf2.view(np.int32)
    assert np.array_equal(np.delete(got2, [4, 5]), np.delete(ref2.blob(), [4, 5]))
    W, C = int(got2[1]), int(got2[2])
    c0 = (16 + 6 * W + 3) // 4 * 4 + 4 * C
    assert C == 6  # every sequence is split (at most 4 ways), two KV heads each
    assert np.all(got2[c0:c0 + C] == 0) and c0 + C <= len(got2)
    p.free()   # must not free the caller's buffer
    assert buf[:4].view(np.int32)[0] == 0x564B4150


def test_decode_rejects_before_launch(lib):
    """Argument errors return before touching CUDA (this host has no GPU)."""
    w = workloads.make_custom(seq_lens=[10, 20], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=4)
    s = _shape(w)
    plan = binding.Plan(s, w.seq_lens, 152)
    fake = ctypes.c_void_p(0x10000)   # aligned, never dereferenced: the calls below fail earlier
    null = ctypes.c_void_p(0)
    args = lambda **o: [o.get(k, fake) for k in ("q", "kp", "vp", "bt", "sl")]
    # null pointer
    r = lib.pa_decode_attention(ctypes.byref(s), ctypes.byref(plan.c), *args(q=null),
                                ctypes.c_float(0.1), fake, fake, plan.c.workspace_bytes, fake, None)
    assert r == 1
    # misaligned q
    r = lib.pa_decode_attention(ctypes.byref(s), ctypes.byref(plan.c), *args(q=ctypes.c_void_p(0x10002)),
                                ctypes.c_float(0.1), fake, fake, plan.c.workspace_bytes, fake, None)
    assert r == 1
    # workspace too small
    r = lib.pa_decode_attention(ctypes.byref(s), ctypes.byref(plan.c), *args(), ctypes.c_float(0.1),
                                fake, fake, plan.c.workspace_bytes - 1, fake, None)
    assert r == 3
    # non-finite scale
    r = lib.pa_decode_attention(ctypes.byref(s), ctypes.byref(plan.c), *args(),
                                ctypes.c_float(float("nan")), fake, fake, plan.c.workspace_bytes, fake, None)
    assert r == 1
    # plan made for another shape
    s2 = binding.make_shape(2, 4, 2, 64, 16, w.max_pages_per_seq + 1, w.num_pages)
    r = lib.pa_decode_attention(ctypes.byref(s2), ctypes.byref(plan.c), *args(), ctypes.c_float(0.1),
                                fake, fake, plan.c.workspace_bytes, fake, None)
    assert r == 8
    # upload into a too-small workspace
    assert lib.pa_plan_upload(ctypes.byref(plan.c), fake, plan.c.workspace_bytes - 1, None) == 3
    # append with an unsupported head_dim
    s3 = binding.make_shape(2, 4, 2, 80, 16, 4, 8)
    assert lib.pa_kv_append(ctypes.byref(s3), fake, fake, fake, fake, fake, fake, fake, None) == 2


def test_empty_batch_is_a_no_op(lib):
    s = binding.make_shape(0, 4, 2, 64, 16, 4, 8)
    plan = binding.Plan(s, np.zeros(0, np.int32), 152)
    assert plan.c.num_work_items == 0
    fake = ctypes.c_void_p(0x10000)
    assert lib.pa_decode_attention(ctypes.byref(s), ctypes.byref(plan.c), fake, fake, fake, fake,
                                   fake, ctypes.c_float(0.1), fake, fake, 1 << 20, fake, None) == 0
    assert lib.pa_kv_append(ctypes.byref(s), fake, fake, fake, fake, fake, fake, fake, None) == 0


def test_prefill_plan_tiles_cover_every_row_once(lib):
    lens = [37, 100, 5, 640, 0]
    qls = [37, 5, 0, 640, 0]
    for hq, hkv in ((4, 2), (8, 8), (32, 4)):
        s = binding.make_shape(len(lens), hq, hkv, 64, 16, 40, 100)
        plan = binding.PrefillPlan(s, lens, qls)
        blob = plan.blob()
        assert blob[0] == 0x564B4650 and blob[1] == plan.c.num_tiles and blob[3] == sum(qls)
        n = int(blob[1])
        tiles = blob[16:16 + 4 * n].reshape(n, 4)
        cu = blob[16 + 4 * n:16 + 4 * n + len(lens) + 1]
        assert cu.tolist() == np.concatenate([[0], np.cumsum(qls)]).tolist()
        G = hq // hkv
        seen = set()
        for b, g, tok0, ntok in tiles:
            assert 1 <= ntok <= int(blob[8]) // G and tok0 + ntok <= qls[b]
            for i in range(tok0, tok0 + ntok):
                seen.add((int(b), int(g), i))
        assert seen == {(b, g, i) for b in range(len(lens)) for g in range(hkv)
                        for i in range(qls[b])}
        # longest stream first (a tile's time follows the keys it streams)
        span = [lens[b] - qls[b] + tok0 + ntok for b, g, tok0, ntok in tiles]
        assert all(x >= y for x, y in zip(span, span[1:]))
    s = binding.make_shape(2, 4, 2, 64, 16, 8, 20)
    with pytest.raises(binding.PagedAttnError) as e:
        binding.PrefillPlan(s, [10, 20], [11, 1])      # more queries than cached tokens
    assert e.value.code == 1


def test_plans_from_many_host_threads_agree(lib):
    """pa_plan keeps no shared state but a plan-id counter: plans made at once
    on several host threads equal the plan made alone (ids aside)."""
    import threading
    lens = np.random.default_rng(3).integers(1, 4000, size=160).astype(np.int32)
    s = binding.make_shape(len(lens), 32, 8, 128, 16, 256, 8192)
    ref = binding.Plan(s, lens, 152, 0).blob()
    out, errors = [], []

    def work():
        try:
            for _ in range(20):
                b = binding.Plan(s, lens, 152, 0).blob()
                b[4:6] = ref[4:6]   # the plan id stamp differs by design
                out.append(b)
        except Exception as e:   # surfaced below
            errors.append(e)
    threads = [threading.Thread(target=work) for _ in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors
    assert len(out) == 160 and all(np.array_equal(b, ref) for b in out)


def test_plan_options_zeroed_equal_the_plain_plan(lib):
    """pa_plan_ex with a zeroed options struct makes pa_plan's task list, and
    copies the per-call fields (all zero: the defaults) into the plan."""
    for cfg in (2, 4, 5):
        w = workloads.make_config(cfg)
        ref = binding.Plan(_shape(w), w.seq_lens, 152, w.forced_splits)
        p = binding.Plan(_shape(w), w.seq_lens, 152, w.forced_splits,
                         options=binding.plan_options())
        assert np.array_equal(np.delete(p.blob(), [4, 5]), np.delete(ref.blob(), [4, 5]))
        assert (p.c.merge, p.c.l2_prefetch_pages, p.c.l2_prefetch_ctas, p.c.wait_limit_ns,
                p.c.early_kv) == (0,) * 5
        assert p.c.owns_blob == 1


def test_plan_options_shape_the_task_list(lib):
    w = workloads.make_config(4)
    s = _shape(w)
    base = binding.Plan(s, w.seq_lens, 152)
    # finer minimum chunks and more waves: more, shorter splits
    fine = binding.Plan(s, w.seq_lens, 152, options=binding.plan_options(min_chunk_pages=16, waves=4))
    assert fine.c.num_work_items > base.c.num_work_items and fine.c.chunk_pages < base.c.chunk_pages
    check_plan_covers(w, fine)
    # the skewed mix bundles its short tasks by default; bundle_max_pages < 0 never does
    w5 = workloads.make_config(5)
    b5 = binding.Plan(_shape(w5), w5.seq_lens, 152)
    assert b5.c.num_shared_ctas < b5.c.num_work_items
    nb = binding.Plan(_shape(w5), w5.seq_lens, 152, options=binding.plan_options(bundle_max_pages=-1))
    assert nb.c.num_shared_ctas == nb.c.num_work_items == nb.c.num_ctas
    check_plan_covers(w5, nb)
    # bundle_waves < 0 bundles short tasks at any task count: workload 3's
    # 1536 tasks (below 3 waves of CTAs) go four to a CTA, one per warp
    w3 = workloads.make_config(3)
    b3 = binding.Plan(_shape(w3), w3.seq_lens, 152)
    assert b3.c.num_shared_ctas == b3.c.num_work_items == b3.c.num_ctas
    a3 = binding.Plan(_shape(w3), w3.seq_lens, 152,
                      options=binding.plan_options(bundle_waves=-1, bundle_max_pages=64))
    assert a3.c.num_shared_ctas == 0 and a3.c.num_ctas == (a3.c.num_work_items + 3) // 4
    check_plan_covers(w3, a3, bundle_max=64)
    # the per-call fields are carried by the plan, in a caller buffer too
    buf = np.zeros(base.c.blob_bytes, np.uint8)
    o = binding.plan_options(merge="combine", l2_prefetch_pages=32, l2_prefetch_ctas=7,
                             wait_limit_ns=12345, early_kv=1)
    p = binding.Plan(s, w.seq_lens, 152, host_buffer=buf, options=o)
    assert p.c.owns_blob == 0 and p.c.host_blob == buf.ctypes.data
    assert (p.c.merge, p.c.l2_prefetch_pages, p.c.l2_prefetch_ctas, p.c.wait_limit_ns,
            p.c.early_kv) == (binding.PA_MERGE_COMBINE_KERNEL, 32, 7, 12345, 1)
    # early_kv changes when the kernel reads, not the task list
    assert np.array_equal(np.delete(p.blob(), [4, 5]), np.delete(base.blob(), [4, 5]))


@pytest.mark.parametrize("bad", [dict(merge=2), dict(merge=-1), dict(l2_prefetch_pages=33),
                                 dict(waves=-1), dict(waves=65), dict(min_chunk_pages=-1),
                                 dict(bundle_waves=65), dict(early_kv=2), dict(early_kv=-1)])
def test_plan_options_out_of_range_are_refused(lib, bad):
    w = workloads.make_custom(seq_lens=[10, 20], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=6)
    with pytest.raises(binding.PagedAttnError) as e:
        binding.Plan(_shape(w), w.seq_lens, 152, options=binding.plan_options(**bad))
    assert e.value.code == 1, bad


@pytest.mark.parametrize("field,value", [("merge", 5), ("q8_stages", 4), ("early_kv", 2)])
def test_decode_refuses_a_plan_with_bad_call_fields(lib, field, value):
    """A plan edited after pa_plan_ex into an out-of-range call field is
    refused before any launch."""
    w = workloads.make_custom(seq_lens=[10, 20], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=7)
    s = _shape(w)
    plan = binding.Plan(s, w.seq_lens, 152)
    setattr(plan.c, field, value)
    fake = ctypes.c_void_p(0x10000)
    r = lib.pa_decode_attention(ctypes.byref(s), ctypes.byref(plan.c), fake, fake, fake, fake, fake,
                                ctypes.c_float(0.1), fake, fake, plan.c.workspace_bytes, fake, None)
    assert r == 8


def test_prefill_plan_rows_per_tile_option(lib):
    lens, qls = [300, 40], [200, 40]
    s = binding.make_shape(2, 8, 2, 128, 16, 32, 64)
    d = binding.PrefillPlan(s, lens, qls)
    assert d.c.rows_per_tile == 128 and d.blob()[8] == 128 and d.c.wait_limit_ns == 0
    p = binding.PrefillPlan(s, lens, qls, rows_per_tile=64, wait_limit_ns=99)
    assert p.c.rows_per_tile == 64 and p.blob()[8] == 64 and p.c.wait_limit_ns == 99
    assert p.c.num_tiles > d.c.num_tiles   # half the rows per tile: about twice the tiles
    with pytest.raises(binding.PagedAttnError) as e:
        binding.PrefillPlan(s, lens, qls, rows_per_tile=96)
    assert e.value.code == 1


def test_library_reads_no_environment():
    """Tuning and test knobs come through the plan options, not from
    process-global environment variables."""
    import os
    import re
    csrc = os.path.join(os.path.dirname(binding.__file__), "csrc")
    for name in os.listdir(csrc):
        text = open(os.path.join(csrc, name), errors="replace").read()
        assert not re.search(r"\b(secure_)?getenv\s*\(", text), name


def test_static_entry_checks_before_anything_is_queued(lib):
    """pa_decode_attention_static makes pa_decode_attention's checks, in its
    order, and returns before its first CUDA call when one fails (this host
    has no GPU, so a call that got further would fail differently)."""
    w = workloads.make_custom(seq_lens=[10, 20], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=8)
    s = _shape(w)
    plan = binding.Plan(s, w.seq_lens, 152, 2)
    fake = ctypes.c_void_p(0x10000)
    call = lambda shape, pl, scale=0.1, q=fake: lib.pa_decode_attention_static(
        ctypes.byref(shape), ctypes.byref(pl.c), q, fake, fake, fake, fake, ctypes.c_float(scale),
        fake, fake, None)
    assert call(s, plan, scale=float("nan")) == 1
    assert call(s, plan, scale=float("inf")) == 1
    assert call(s, plan, q=ctypes.c_void_p(0x10008)) == 1
    other = binding.make_shape(2, 4, 2, 64, 16, w.max_pages_per_seq + 1, w.num_pages)
    assert call(other, plan) == 8
    # batch 0 with a plan of another shape: PA_ERR_PLAN, as pa_decode_attention
    s0 = binding.make_shape(0, 4, 2, 64, 16, 4, 8)
    assert call(s0, plan) == 8
    r = lib.pa_decode_attention(ctypes.byref(s0), ctypes.byref(plan.c), fake, fake, fake, fake,
                                fake, ctypes.c_float(0.1), fake, fake, 1 << 20, fake, None)
    assert r == 8
    # batch 0 with its own plan: nothing to do
    p0 = binding.Plan(s0, np.zeros(0, np.int32), 152)
    assert call(s0, p0) == 0


def test_one_wave_split_rule(lib):
    """The automatic split size is the average page load of a resident CTA,
    never under 48 pages: chunk = max(48, ceil(units / (SMs * r))) with r = 4
    resident CTAs per SM for every group size and head_dim (every split
    kernel stops at four, by registers and shared memory alike), the same r
    that option waves = 2 halves.  Every sequence is cut into
    ceil(pages / chunk) ranges of at most chunk pages."""
    # workload 4: every (sequence, KV head) is shorter than that load, so no split
    w4 = workloads.make_config(4)
    p4 = binding.Plan(_shape(w4), w4.seq_lens, 152)
    assert p4.c.num_groups == 0 and p4.c.num_work_items == w4.batch * w4.num_kv_heads
    rng = np.random.default_rng(5)
    for trial in range(16):
        B = int(rng.integers(1, 48))
        lens = rng.integers(1, 24000, size=B).astype(np.int32)
        hkv = int(rng.choice([1, 2, 8, 32]))
        hq = hkv * int(rng.choice([1, 2, 4, 8]))
        d = int(rng.choice([64, 128]))
        max_pages = int(lens.max() + 15) // 16
        shape = binding.make_shape(B, hq, hkv, d, 16, max_pages, max_pages * B)
        # only the plan is made: the shape and lengths, no pools
        w = types.SimpleNamespace(page_size=16, batch=B, num_kv_heads=hkv, seq_lens=lens)
        sms = int(rng.choice([8, 40, 152]))
        p1 = binding.Plan(shape, lens, sms)
        p2 = binding.Plan(shape, lens, sms, options=binding.plan_options(waves=2))
        units = int(sum(max(1, (int(L) + 15) // 16) for L in lens)) * hkv
        fits = [r for r in range(1, 17)
                if p1.c.chunk_pages == max(48, -(-units // (sms * r)))
                and p2.c.chunk_pages == max(48, -(-units // (2 * sms * r)))]
        assert 4 in fits, (trial, hq // hkv, d, p1.c.chunk_pages, p2.c.chunk_pages, units, sms)
        items, _ = check_plan_covers(w, p1)
        assert np.all(items[:, 3] - items[:, 2] <= p1.c.chunk_pages)
        per_seq = {}
        for b, hw, lo, hi in items:
            per_seq[(int(b), int(hw) & 0xFFFF)] = per_seq.get((int(b), int(hw) & 0xFFFF), 0) + 1
        for (b, h), n in per_seq.items():
            pages = max(1, (int(lens[b]) + 15) // 16)
            assert n == min(1024, -(-pages // p1.c.chunk_pages)) or (int(lens[b]) == 0 and n == 1)


def test_q8_stage_rule(lib):
    """The 8-bit kernel's page stages: 3 when every CTA is resident at once
    (152 SMs x 4); otherwise 2 when the tasks average at most 12 pages per
    warp, else 3; the option forces either; other values are refused."""
    want = {1: 3, 2: 3, 3: 2, 4: 3, 5: 2}
    for cfg, ns in want.items():
        w = workloads.make_config(cfg)
        p = binding.Plan(_shape(w), w.seq_lens, 152, w.forced_splits)
        items, _ = check_plan_covers(w, p)
        pages = int(np.sum(items[:, 3] - items[:, 2]))
        n_shared = p.c.num_shared_ctas
        warps = n_shared * 4 + (p.c.num_work_items - n_shared)
        rule = 3 if p.c.num_ctas <= 152 * 4 else (2 if pages <= 12 * warps else 3)
        assert p.c.q8_stages == ns == rule, (cfg, pages, warps, p.c.num_ctas)
        for forced in (2, 3):
            f = binding.Plan(_shape(w), w.seq_lens, 152, w.forced_splits,
                             options=binding.plan_options(q8_stages=forced))
            assert f.c.q8_stages == forced
    w = workloads.make_config(4)
    for bad in (1, 4, -1):
        with pytest.raises(binding.PagedAttnError):
            binding.Plan(_shape(w), w.seq_lens, 152, options=binding.plan_options(q8_stages=bad))
