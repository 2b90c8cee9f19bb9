"""The multi-token oracle over every row of a large workload, spread over a
pool of processes started with spawn (safe in a test process that already
holds a CUDA context; a forked child of one can hang).  Each process rebuilds
the seeded workload from its recipe, so no large array crosses a process
boundary, and takes every n-th query row (all heads), which balances the
causal spans.  The rows are computed by oracle.prefill_attention as they
would be in one process; this only divides the work."""

from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _build(recipe):
    from paged_kv_decode_24_gb300 import workloads
    kind, arg = recipe
    if kind == "prefill_config":
        return workloads.make_prefill_config(arg)
    if kind == "custom":
        return workloads.make_custom(**arg)
    raise ValueError(kind)


def _rows(job):
    recipe, share, nshare = job
    import oracle
    w = _build(recipe)
    kp, vp = oracle.kv_append_tokens(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                     w.seq_lens, w.q_lens)
    mine = list(range(share, w.q.shape[0], nshare))
    rows = [(r, h) for r in mine for h in range(w.num_q_heads)]
    out = oracle.prefill_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.q_lens, w.scale,
                                   rows=rows)
    return mine, out[mine]


def prefill_all(recipe, processes=None):
    """float64 [T][Hq][D]: every output of the workload the recipe builds
    (("prefill_config", n) or ("custom", make_custom keyword arguments))."""
    n = processes or max(1, min(16, len(os.sched_getaffinity(0))
                                if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1))
    # one BLAS thread per process (the children copy the environment when
    # they start): n processes of many threads each would oversubscribe
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ.update({k: "1" for k in keys})
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            parts = pool.map(_rows, [(recipe, i, n) for i in range(n)])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    T = sum(len(m) for m, _ in parts)
    first = parts[0][1]
    out = np.full((T,) + first.shape[1:], np.nan, np.float64)
    for mine, vals in parts:
        out[mine] = vals
    return out
