"""GPU: plans made with early_kv (the split kernel reads seq_lens and the
block table and starts its first page copies before it waits for the kernel
ahead of it in the stream; q and the new rows come after the wait).

A chain of layer calls, each over its own layer's cache, is queued behind a
spin kernel so that the launches run back to back and each layer's kernel
starts while the one ahead of it still runs (programmatic dependent launch):
- every layer's output and appended pool rows match the float64 oracle;
- when each layer's q is the output of the layer ahead (written by the
  kernel still running when the next starts), the outputs are bit-identical
  to the same chain run without early_kv.
The same chain captured in a CUDA graph (programmatic edges between the
kernels) and replayed matches the oracle too.
All five split kernels take part: fp16 and bf16 CUDA-core (MHA) and tensor-core
(GQA) kernels and the 8-bit kernel over INT8 and FP8 caches, with the split
merge inside the split kernel or in the separate combine kernel.
"""

from __future__ import annotations

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

LAYERS = 6
LENS = [1900, 37, 700, 1, 16, 1333, 250, 0, 1024, 511]


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    return lib


# (cache, element type, q heads, KV heads, head_dim, forced splits, merge)
CASES = [
    ("fp16", "fp16", 16, 16, 128, 0, "split"),     # CUDA-core kernel, MHA
    ("fp16", "bf16", 8, 8, 64, 3, "combine"),     # CUDA-core kernel, combine kernel
    ("fp16", "fp16", 32, 8, 128, 4, "split"),      # tensor-core kernel, GQA-4
    ("fp16", "bf16", 16, 2, 128, 0, "combine"),    # tensor-core kernel, GQA-8
    ("int8", "fp16", 32, 8, 128, 2, "split"),      # 8-bit kernel
    ("fp8", "fp16", 16, 16, 128, 0, "split"),      # 8-bit kernel, MHA
    ("fp8", "fp16", 8, 4, 64, 5, "combine"),
]


def _ids(c):
    return f"{c[0]}-{c[1]}_G{c[2] // c[3]}_D{c[4]}_s{c[5]}_{c[6]}"


def _layers(case):
    kv, dtype, hq, hkv, d, splits, _ = case
    cache = kv if kv in ("int8", "fp8") else "fp16"
    return [workloads.make_custom(seq_lens=LENS, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                  seed=9100 + 17 * l, forced_splits=splits, kv=cache, dtype=dtype,
                                  poison=True)
            for l in range(LAYERS)]


def _call(dd, q, out):
    """The layer's pa_append_decode_attention (its cache's form) with q."""
    saved, dd.q = dd.q, q
    try:
        return (dd.append_decode8 if dd.kv in ("int8", "fp8") else dd.append_decode)(out)
    finally:
        dd.q = saved


def _chain(dds, plan_of, qs, outs):
    """Every layer's call, queued behind a spin kernel on the current stream."""
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2000 * 2100))   # ~2 ms: the host queues the whole chain meanwhile
    for l, dd in enumerate(dds):
        dd.plan_obj, dd.workspace = plan_of
        _call(dd, qs[l], outs[l])
    torch.cuda.synchronize()


def _same_pool(got, host):
    """Device pool against the oracle's: the same bits, except that the NaN
    of a poisoned row may carry another payload (the device pools were
    converted to bf16 on the GPU, the oracle's on the host)."""
    ref = torch.from_numpy(np.ascontiguousarray(host)).to(got.dtype)
    if not got.dtype.is_floating_point:
        return torch.equal(got, ref)
    gn, rn = torch.isnan(got), torch.isnan(ref)
    bits = torch.int16 if got.element_size() == 2 else torch.int32
    return torch.equal(gn, rn) and torch.equal(got[~gn].view(bits), ref[~rn].view(bits))


def _plan(dds, case, early):
    """One plan and workspace for every layer (same lengths)."""
    dds[0].plan_obj = None
    dds[0].make_plan(merge=case[6], early_kv=int(early))
    assert dds[0].plan_obj.c.early_kv == int(early)
    return dds[0].plan_obj, dds[0].workspace


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_layer_chain_early_kv_matches_oracle(case):
    ws = _layers(case)
    dds = [DeviceDecode(w) for w in ws]
    plan = _plan(dds, case, early=True)
    outs = [torch.empty_like(dd.q) for dd in dds]
    _chain(dds, plan, [dd.q for dd in dds], outs)
    for l, (w, dd) in enumerate(zip(ws, dds)):
        assert dd.read_status() == 0, (case, l)
        if w.kv in ("int8", "fp8"):
            want, (kc, vc, ks, vs) = oracle_append_decode(w)
            pools = [(dd.k_codes, kc), (dd.v_codes, vc), (dd.k_scales, ks), (dd.v_scales, vs)]
        else:
            kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                      w.seq_lens)
            want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
            pools = [(dd.k_pages, kp), (dd.v_pages, vp)]
        assert_close(outs[l].float().cpu().numpy(), want, f"early_kv chain {case} layer {l}",
                     dtype=w.dtype)
        for dev, host in pools:
            assert _same_pool(dev.cpu(), host), (case, l)


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_q_from_the_layer_ahead_is_read_after_the_wait(case):
    """Layer l + 1's q is layer l's output buffer, written by the kernel
    that may still run when layer l + 1's starts: with early_kv every output
    is bit-identical to the chain without it, and layer 0's matches the
    oracle."""
    ws = _layers(case)
    dds = [DeviceDecode(w) for w in ws]
    bufs = [dds[0].q.clone()] + [torch.empty_like(dds[0].q) for _ in range(LAYERS)]
    results = {}
    for early in (False, True):
        plan = _plan(dds, case, early)
        for b in bufs[1:]:
            b.fill_(float("nan"))
        _chain(dds, plan, bufs[:-1], bufs[1:])
        for l, dd in enumerate(dds):
            assert dd.read_status() == 0, (case, early, l)
        results[early] = [b.clone() for b in bufs[1:]]
    for l in range(LAYERS):
        a, b = results[False][l], results[True][l]
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (case, l)
    w = ws[0]
    if w.kv in ("int8", "fp8"):
        want, _ = oracle_append_decode(w)
    else:
        kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                  w.seq_lens)
        want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
    assert_close(results[True][0].float().cpu().numpy(), want, f"early_kv layer 0 {case}",
                 dtype=w.dtype)


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[4]], ids=_ids)
def test_layer_chain_early_kv_in_a_captured_graph(case):
    """The chain captured once in a CUDA graph (programmatic edges between
    the layers' kernels, as the bench runs it) and replayed twice: every
    layer's output and appended rows match the oracle (the append writes the
    same rows again on the second replay)."""
    ws = _layers(case)
    dds = [DeviceDecode(w) for w in ws]
    plan, work = _plan(dds, case, early=True)
    outs = [torch.empty_like(dd.q) for dd in dds]
    for l, dd in enumerate(dds):   # one eager pass: one-time kernel setup outside capture
        dd.plan_obj, dd.workspace = plan, work
        _call(dd, dd.q, outs[l])
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for l, dd in enumerate(dds):
            _call(dd, dd.q, outs[l])
    for _ in range(2):
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
    for l, (w, dd) in enumerate(zip(ws, dds)):
        assert dd.read_status() == 0, (case, l)
        if w.kv in ("int8", "fp8"):
            want, (kc, vc, ks, vs) = oracle_append_decode(w)
            pools = [(dd.k_codes, kc), (dd.v_codes, vc), (dd.k_scales, ks), (dd.v_scales, vs)]
        else:
            kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                      w.seq_lens)
            want = oracle.decode_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.scale)
            pools = [(dd.k_pages, kp), (dd.v_pages, vp)]
        assert_close(outs[l].float().cpu().numpy(), want, f"early_kv graph {case} layer {l}",
                     dtype=w.dtype)
        for dev, host in pools:
            assert _same_pool(dev.cpu(), host), (case, l)
