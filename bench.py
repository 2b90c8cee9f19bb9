"""Benchmark: decode attention over a paged KV cache on one GB300 (or N replicas).

One step is one layer's decode attention over one batch:
    pa_append_decode_attention (one kernel: the append of the new token
    fused into the split kernel, whose last split per group merges the
    partials by their log-sum-exp),
and once per 32-layer model step pa_plan_upload of that step's plan, inside
the timed region.  pa_plan makes each model step's plan on the host while
the GPU runs the model step before it (the plan depends only on seq_lens,
which every layer shares).  Inputs are synthetic and seeded, with the
shapes of the five workloads in paged_kv_decode_24_gb300/workloads.py.  The
headline is workload 4 (LLaMA-3-8B heads, batch 160, GQA-4, the largest);
workloads 2, 3 and 5, and workload 4 over the INT8 and FP8 caches, are timed
the same way in the same run and reported under per_config (8-bit lines count
8-bit bytes).

Each model step (32 layer steps) is one CUDA graph: the plan upload, then
the 32 layers' calls back to back; K layer steps are timed exactly (a shorter
graph covers K mod 32).  A spin kernel queued before the start event holds
the stream while the host queues the timed graphs, so the events time the
device's work and not the host's launch latency.

The JSON line reports:
  value         KV-read GB/s of the whole job (K and V bytes of every attended
                token / device time per step), all ranks together
  ms_per_step   device time per layer step (CUDA events, max over ranks)
  roofline      the fused call (one split kernel launch) against the
                measured HBM copy bandwidth: its mean duration over the timed
                region; us_per_launch_isolated is one call alone (own graph)
  e2e           the same metric with host buffers: per-step inputs copied
                from pinned host memory and the output read back
  cpu_baseline  the float64 oracle on one host core, on a bounded sample;
                cpu_baseline_all_cores runs it on every core at once
  plan_host_us  one pa_plan call on the host (not part of the device timing)
  append_us     pa_kv_append alone, as its own launch (the step fuses it)
  per_config    the other workloads' (and the 8-bit caches') µs per step,
                GB/s and roofline fraction

Each of the 32 layers has its own KV cache (distinct device memory, 2-29 GiB
in total), so L2 never holds the pages a step reads.

--kv int8 runs the same steps over the INT8 cache (codes with one fp32 scale
per row) through pa_append_decode_attention_q8, --kv fp8 over the FP8 (E4M3)
cache through pa_append_decode_attention_fp8; value and roofline then count
the 8-bit rows' bytes (D + 4 per row and tensor).

--impl reference times the float64 CPU oracle (the only reference this
method has) on the same workload, metric and unit.
"""

from __future__ import annotations

import os as _os
import sys as _sys

if "--impl" in _sys.argv and "reference" in _sys.argv:
    # the oracle runs single-threaded, as in the CPU baseline; set before numpy loads
    for _k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        _os.environ[_k] = "1"

import argparse
import copy
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention µs/step and KV-read GB/s as % of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4, choices=[1, 2, 3, 4, 5],
                    help="the headline workload (default 4: LLaMA-3-8B heads, batch 160, the "
                         "largest)")
    ap.add_argument("--also", type=parse_also, default=None,
                    help="decode: other workloads timed in the same run and reported under "
                         "per_config, each a workload id or id-kv for an 8-bit cache (default "
                         "2,3,5,4-int8,4-fp8 with the default headline; '' for none)")
    ap.add_argument("--merge", choices=["split", "combine"], default="split",
                    help="decode: merge split partials in the split kernel (one launch) or in "
                         "a separate combine kernel (plan option merge)")
    ap.add_argument("--plan", default="",
                    help="decode: plan options as name=value pairs, comma-separated "
                         "(min_chunk_pages, waves, bundle_max_pages, bundle_waves, "
                         "l2_prefetch_pages, l2_prefetch_ctas); for experiments")
    ap.add_argument("--early-kv", choices=["on", "off"], default="on",
                    help="decode: plan option early_kv; each layer's call reads its own "
                         "layer's cache, which no kernel still running writes, so its first "
                         "page copies may start before the wait on the layer ahead (on)")
    ap.add_argument("--upload", choices=["ahead", "inline"], default="ahead",
                    help="decode: each model step's graph uploads the next step's plan into a "
                         "second workspace while its layers run (ahead), or its own plan before "
                         "its first layer (inline)")
    ap.add_argument("--decode-rows", choices=["tiles", "decode-call"], default="tiles",
                    help="prefill: sequences with one query token go through the multi-token "
                         "kernel's tiles like the others (tiles), or through "
                         "pa_append_decode_attention on a second stream while the rest run "
                         "(decode-call)")
    ap.add_argument("--prefill-rows", type=int, choices=[128, 64], default=128,
                    help="prefill: query rows per tile, 128 for the tcgen05 kernel, 64 for the "
                         "mma.sync kernel (plan option rows_per_tile)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--oracle-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-offset", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-stride", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kv", choices=["fp16", "int8", "fp8"], default="fp16",
                    help="KV-cache type: 16-bit elements, or INT8 codes or FP8 (E4M3) bytes with "
                         "per-row fp32 scales")
    ap.add_argument("--op", choices=["decode", "swap", "prefill"], default="decode",
                    help="decode: the decode step; swap: KV block swap-out + swap-in "
                         "(pa_copy_blocks) of a quarter of the workload's sequences; prefill: "
                         "several query tokens per sequence (--config 1 or 2 picks the "
                         "multi-token workload)")
    ap.add_argument("--dtype", choices=["fp16", "bf16"], default="fp16",
                    help="element type of q, K, V and out (the 8-bit caches take fp16)")
    ap.add_argument("--layers", type=int, default=MODEL_LAYERS,
                    help="per-layer KV caches; fewer only to shrink profiler captures")
    ap.add_argument("--splits", type=int, default=None,
                    help="decode: force this split count per sequence in place of the "
                         "workload's own (0 = the planner's choice); for experiments")
    args = ap.parse_args()
    if args.also is None:
        args.also = (list(EXTRA_CONFIGS) if args.config == 4 and args.op == "decode" and
                     args.kv == "fp16" and args.dtype == "fp16" else [])
    return args


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)

def oracle_sample(w, budget_s, offset=0, stride=1):
    """Run the float64 oracle's attention on whole sequences (every head)
    until about ``budget_s`` seconds pass, taking sequences offset,
    offset + stride, ... of the longest-first order (cycling).  Returns
    (seconds, KV bytes covered, description).  The oracle's append is left
    out: it copies whole pools functionally, which says nothing about the
    method."""
    import oracle
    q8 = w.k_codes is not None
    row = w.head_dim + 4 if q8 else 2 * w.head_dim
    order = list(np.argsort(-w.seq_lens, kind="stable"))   # longest first, cycling
    t0 = time.perf_counter()
    kv = 0
    seqs = 0
    i = offset
    while True:
        b = int(order[i % len(order)])
        i += stride
        sub_bt = w.block_table[b:b + 1]
        sub_l = w.seq_lens[b:b + 1]
        if q8 and w.kv == "fp8":
            oracle.decode_attention_fp8(w.q[b:b + 1], w.k_codes, w.v_codes, w.k_scales,
                                        w.v_scales, sub_bt, sub_l, w.scale)
        elif q8:
            oracle.decode_attention_q8(w.q[b:b + 1], w.k_codes, w.v_codes, w.k_scales,
                                       w.v_scales, sub_bt, sub_l, w.scale)
        else:
            oracle.decode_attention(w.q[b:b + 1], w.k_pages, w.v_pages, sub_bt, sub_l, w.scale)
        kv += int(sub_l[0]) * w.num_kv_heads * 2 * row
        seqs += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s and seqs >= 1:
            break
    return dt, kv, f"{seqs} whole sequences (all heads), longest first"


def oracle_worker(args):
    from paged_kv_decode_24_gb300 import workloads
    w = workloads.make_config(args.config, kv=args.kv, dtype=args.dtype)
    dt, kv, desc = oracle_sample(w, args.cpu_seconds, args.oracle_offset, args.oracle_stride)
    print(json.dumps({"seconds": dt, "kv_bytes": kv, "sample": desc}))


def run_oracle_subprocess(cfg, seconds, kv="fp16", dtype="fp16"):
    """The oracle in a fresh single-threaded process (started by exec, so no
    CUDA state is shared)."""
    from paged_kv_decode_24_gb300 import workloads
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-worker", "--config",
                        str(cfg), "--cpu-seconds", str(seconds), "--kv", kv, "--dtype", dtype],
                       capture_output=True, text=True,
                       env=env, timeout=600)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    res = json.loads(r.stdout.strip().splitlines()[-1])
    gbs = res["kv_bytes"] / res["seconds"] / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{workloads.CONFIG_NAMES[cfg]} ({kv} cache, {dtype}): {res['sample']}, "
                      f"{res['seconds']:.1f} s of float64 numpy"}


def run_oracle_all_cores(cfg, seconds, kv="fp16", dtype="fp16"):
    """The oracle on every core this process may use: one single-threaded
    process per core (started by exec, no CUDA state), each on its own share
    of the sequences (offset i, stride n), all for about ``seconds``.  GB/s =
    the KV bytes of all of them / the longest one's time."""
    from paged_kv_decode_24_gb300 import workloads
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    procs = [subprocess.Popen([sys.executable, os.path.abspath(__file__), "--oracle-worker",
                               "--config", str(cfg), "--cpu-seconds", str(seconds), "--kv", kv,
                               "--dtype", dtype, "--oracle-offset", str(i),
                               "--oracle-stride", str(n)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env)
             for i in range(n)]
    res = []
    for pr in procs:
        out, err = pr.communicate(timeout=600)
        if pr.returncode != 0:
            raise RuntimeError(err[-2000:])
        res.append(json.loads(out.strip().splitlines()[-1]))
    kvb = sum(r["kv_bytes"] for r in res)
    dt = max(r["seconds"] for r in res)
    return {"value": kvb / dt / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{workloads.CONFIG_NAMES[cfg]} ({kv} cache, {dtype}): {n} single-threaded processes, "
                      f"sequences dealt round-robin, {dt:.1f} s of float64 numpy each"}


# ---------------------------------------------------------------------------
# device helpers

def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Sources a split-decode kernel family and its launch are built from: the
# family's kernel files, the device helpers, the planner that sets the grid,
# and the C-ABI that fills the launch parameters.
DECODE_COMMON = ("api.cu", "device_common.cuh", "elem.cuh", "split_launch.cuh",
                 "split_merge.cuh", "pa_internal.h", "launch.h", "plan.cpp")
DECODE_FAMILY = {"cc": ("decode_kernel.cuh", "decode_d64.cu", "decode_d128.cu"),
                 "tc": ("decode_kernel.cuh", "decode_tc.cuh", "decode_tc_d64.cu",
                        "decode_tc_d128.cu"),
                 "q8": ("decode_kernel.cuh", "decode_tc.cuh", "decode_q8.cuh", "quant_common.cuh",
                        "decode_q8_d64.cu", "decode_q8_d128.cu"),
                 "f8": ("decode_kernel.cuh", "decode_tc.cuh", "decode_q8.cuh", "quant_common.cuh",
                        "decode_f8_d64.cu", "decode_f8_d128.cu")}


def decode_family(w, kv):
    """The split kernel a workload runs on: INT8 or FP8 cache, CUDA cores
    (MHA) or tensor cores (GQA)."""
    if kv == "int8":
        return "q8"
    if kv == "fp8":
        return "f8"
    return "cc" if w.num_q_heads == w.num_kv_heads else "tc"


def kernel_source_hash(family):
    """Hash of the sources of one split-decode kernel family, stamped on each
    committed DRAM-traffic capture so that a changed kernel reports no stale
    traffic."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_24_gb300", "csrc")
    for name in sorted(DECODE_COMMON + DECODE_FAMILY[family]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(cfg, kv, dtype, family):
    """DRAM bytes per launch of the split kernel from a committed ncu capture,
    only while that kernel family's sources still hash to what was profiled."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except Exception:
        return None
    key = "-".join([str(cfg)] + [x for x in (kv, dtype) if x != "fp16"])   # "4", "4-int8", "4-bf16"
    ent = d.get("configs", {}).get(key)
    if ent is None or ent.get("source_hash") != kernel_source_hash(family):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.proc = None
        self.uuid = uuid

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.uuid:
            cmd.insert(1, f"--id={self.uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
        time.sleep(0.2)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    """Slowest rank's figure: the job finishes when its last replica does."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(kv_bytes_per_rank, ms_per_step, world):
    """Whole-job KV-read GB/s: every replica reads its own batch once per step
    (weak scaling), and a step lasts as long as the slowest rank's."""
    return world * kv_bytes_per_rank / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# our arm

MODEL_LAYERS = 32   # LLaMA-2-7B and LLaMA-3-8B both have 32 decoder layers
HOLD_US = 300       # spin before a timed region: longer than the host needs to queue the region
# timed in the same run as the headline workload, reported per config: other
# workloads, and the headline workload over the 8-bit caches
EXTRA_CONFIGS = ((2, None), (3, None), (5, None), (4, "int8"), (4, "fp8"))


def parse_also(v):
    """'2,3,4-fp8' -> [(2, None), (3, None), (4, 'fp8')]."""
    out = []
    for x in v.split(","):
        x = x.strip()
        if not x:
            continue
        c, _, kv = x.partition("-")
        if kv and kv not in ("int8", "fp8"):
            raise argparse.ArgumentTypeError(f"unknown cache {kv!r} in --also")
        out.append((int(c), kv or None))
    return out


def hold_stream(torch, stream, us=HOLD_US):
    """Keep `stream` busy for about `us` microseconds (torch's spin kernel), so
    that the work queued after it is already on the device when the timed
    region starts: the events then time the device's work, not the host's
    launch latency (the blocking-kernel practice of GPU benchmark harnesses).
    It runs before the start event and is not part of any timing."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2100))   # clock cycles; the SM clock is at most 2.07 GHz


class DecodeBench:
    """One decode workload on the device: its layers' KV caches, the plan and
    workspace, and the model-step CUDA graphs that the timings replay.

    A layer step is pa_append_decode_attention (or its INT8-cache form) over
    that layer's cache.  A model step is one CUDA graph: the plan upload
    (a2), then the layers' calls back to back, as a serving engine issues
    them.  Each model step's plan is made on the host (pa_plan_in, into a
    pinned buffer) while the GPU runs the model step before it: the plan
    depends only on seq_lens, which every layer shares."""

    def __init__(self, args, cfg, rank, dev, stream, num_sms, layers):
        import torch

        from paged_kv_decode_24_gb300 import accounting, binding, workloads
        self.torch, self.binding = torch, binding
        self.args, self.cfg, self.dev, self.stream, self.LAYERS = args, cfg, dev, stream, layers
        self.num_sms = num_sms
        self.q8 = args.kv in ("int8", "fp8")   # an 8-bit cache
        if self.q8 and args.dtype != "fp16":
            raise SystemExit("the 8-bit caches take fp16 q/out")
        w = workloads.make_config(cfg, seed=workloads.SEED_BASE + cfg + 1000 * rank, kv=args.kv,
                                  dtype=args.dtype)
        if args.splits is not None:
            w.forced_splits = max(0, int(args.splits))
        self.w = w
        self.shape = binding.make_shape(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                        w.page_size, w.max_pages_per_seq, w.num_pages, args.dtype)
        self.kv_bytes = w.kv_bytes_int8() if self.q8 else w.kv_bytes()
        self.dec_bytes = (accounting.decode_bytes(w.seq_lens, w.num_q_heads, w.num_kv_heads,
                                                  w.head_dim, w.page_size, kv=args.kv)
                          + accounting.append_bytes(w.batch, w.num_kv_heads, w.head_dim,
                                                    kv=args.kv))
        self.lens_host = np.ascontiguousarray(w.seq_lens)
        to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.elem_t = torch.bfloat16 if args.dtype == "bf16" else torch.float16
        # bf16 workloads hold bf16-exact float32 values: the cast is exact
        to_elem = lambda a: to_dev(a).to(self.elem_t)
        self.q = to_elem(w.q)
        self.k_new = to_elem(w.k_new)
        self.v_new = to_elem(w.v_new)
        self.bt = to_dev(w.block_table)
        self.sl = to_dev(w.seq_lens)
        if self.q8:
            cache0 = (to_dev(w.k_codes), to_dev(w.v_codes), to_dev(w.k_scales), to_dev(w.v_scales))
        else:
            cache0 = (to_elem(w.k_pages), to_elem(w.v_pages))
        # One KV cache per layer, as in the model: every layer's pages are
        # distinct memory, so a layer's reads never hit what the previous
        # layers left in L2.
        self.pools = [cache0] + [tuple(t.clone() for t in cache0) for _ in range(layers - 1)]
        self.cache_bytes = sum(t.numel() * t.element_size() for t in cache0)
        self.step_call = {"int8": binding.append_decode_q8, "fp8": binding.append_decode_fp8}.get(
            args.kv, binding.append_decode)
        self.out = torch.empty_like(self.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

        # The plan: pa_plan_ex with the merge form asked for, into pinned host
        # memory, double-buffered so the host never rewrites a buffer whose
        # upload may still be pending.
        extra = dict(kv.split("=") for kv in args.plan.split(",") if kv.strip())
        fields = {"merge": args.merge, "early_kv": int(args.early_kv == "on")}
        fields.update({k: int(v) for k, v in extra.items()})
        self.opts = binding.plan_options(**fields)
        self.plan0 = binding.Plan(self.shape, self.lens_host, num_sms, w.forced_splits,
                                  options=self.opts)
        self.staging = [torch.empty(int(self.plan0.c.blob_bytes), dtype=torch.uint8).pin_memory()
                        for _ in range(2)]
        self.staged_evt = [torch.cuda.Event(), torch.cuda.Event()]
        # upload "ahead": model step m's graph computes with workspace m % 2
        # and, on a side branch at the same time, uploads step m + 1's plan
        # into the other workspace.  "inline": one workspace, and each graph
        # uploads its own plan before its first layer.
        self.ahead = args.upload == "ahead"
        self.workspaces = [binding.alloc_workspace(self.plan0, dev)
                           for _ in range(2 if self.ahead else 1)]
        self.side_up = torch.cuda.Stream(device=dev)
        self.struct0 = self.plan0.structure()
        self.staged_plans = [None, None]
        self.ready = set()   # model steps whose plan is already in its pinned buffer
        self.m = 0           # the next model step
        self.replan(1)       # both buffers hold a plan before the graphs that upload them
        self.replan(0)       # are captured; model step 0's is the one in use first
        with torch.cuda.stream(stream):
            binding.upload(self.staged_plans[0], self.ws_for(0), stream=stream)
            # a warm-up call (sets kernel attributes) before capture
            self.layer_call(self.pools[0], self.q, self.k_new, self.v_new, self.out,
                            self.ws_for(0), stream=stream)
        stream.synchronize()
        self.launches_per_step = 1 + (1 if args.merge == "combine" and
                                      self.plan0.c.num_groups > 0 else 0)

    def ws_for(self, slot):
        """The workspace model steps of this parity compute with."""
        return self.workspaces[slot] if self.ahead else self.workspaces[0]

    def layer_call(self, pool, qq, kn, vn, o, ws, stream=None):
        """One layer's fused append + decode over that layer's cache."""
        self.step_call(self.shape, self.plan0, qq, kn, vn, *pool, self.bt, self.sl, self.w.scale, o,
                       ws, self.status, stream=stream)

    def upload_in_graph(self, slot):
        """Inside a model step's capture: inline, this step's plan into the
        workspace; ahead, the next step's plan into the other workspace on a
        side branch (joined by join_upload)."""
        if not self.ahead:
            self.binding.upload(self.staged_plans[slot], self.ws_for(0))
            return
        self.side_up.wait_stream(self.stream)
        with self.torch.cuda.stream(self.side_up):
            self.binding.upload(self.staged_plans[1 - slot], self.ws_for(1 - slot))

    def join_upload(self):
        if self.ahead:
            self.stream.wait_stream(self.side_up)

    def replan(self, m):
        """a2 on the host: model step m's plan into pinned buffer m % 2, which
        graph m (inline) or graph m - 1 (ahead) uploads."""
        slot = m % 2
        self.staged_evt[slot].synchronize()   # that buffer's last upload has completed
        plan = self.binding.Plan(self.shape, self.lens_host, self.num_sms, self.w.forced_splits,
                                 host_buffer=self.staging[slot], options=self.opts)
        if plan.structure() != self.struct0:
            raise RuntimeError("plan structure changed; captured graphs would be stale")
        self.staged_plans[slot] = plan
        self.ready.add(m)

    def capture(self, slot, nlayers):
        """One model step: a plan upload and nlayers layers' calls."""
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self.upload_in_graph(slot)
            for l in range(nlayers):
                self.layer_call(self.pools[l], self.q, self.k_new, self.v_new, self.out,
                                self.ws_for(slot))
            self.join_upload()
        return g

    def graphs(self, K):
        full, rem = divmod(K, self.LAYERS)
        gf = [self.capture(i, self.LAYERS) for i in range(2)] if full else []
        gr = [self.capture(i, rem) for i in range(2)] if rem else []
        return gf, gr

    def run_steps(self, nsteps, gfull, grem):
        """nsteps layer steps as model-step graphs.  The host makes model
        step n + 1's plan while the GPU runs step n: inline, right after
        step n is queued; ahead, right before (graph n uploads it)."""
        nf, nr = divmod(nsteps, self.LAYERS)
        sched = [gfull] * nf + ([grem] if nr else [])
        for i, gs in enumerate(sched):
            m = self.m
            read = m + 1 if self.ahead else m   # the plan graph m uploads
            if read not in self.ready:
                self.replan(read)
            gs[m % 2].replay()
            self.staged_evt[read % 2].record(self.stream)
            self.ready.discard(read)
            self.m = m + 1
            if not self.ahead and i + 1 < len(sched):
                self.replan(self.m)

    def time_region(self, K, gfull, grem, world):
        """Device time (ms) of K layer steps between CUDA events on the
        launching stream.  The first model step's plan is made before the
        region, as it would be during the step before it."""
        torch = self.torch
        if not self.ahead and self.m not in self.ready:
            self.replan(self.m)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        hold_stream(torch, self.stream)
        with torch.cuda.stream(self.stream):
            start.record(self.stream)
            self.run_steps(K, gfull, grem)
            end.record(self.stream)
        torch.cuda.synchronize()
        barrier(world)
        self.check_status()
        return start.elapsed_time(end)

    def warm(self, nsteps, gfull, grem):
        with self.torch.cuda.stream(self.stream):
            self.run_steps(nsteps, gfull, grem)
        self.stream.synchronize()
        self.check_status()

    def check_status(self):
        if int(self.status.item()) != 0:
            raise RuntimeError(f"device status {int(self.status.item()):#x}")

    def isolated_us(self):
        """One call alone (its own graph, events around it), over the layers'
        caches in turn so L2 holds none of its pages."""
        torch = self.torch
        n_iso = min(self.LAYERS, 8)
        g1 = []
        for l in range(n_iso):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self.layer_call(self.pools[l], self.q, self.k_new, self.v_new, self.out,
                                self.ws_for(0))
            g1.append(g)
        iso = []
        with torch.cuda.stream(self.stream):
            for i in range(24):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(self.stream)
                g1[i % n_iso].replay()
                b.record(self.stream)
                iso.append((a, b))
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in iso[8:]])) * 1e3

    def e2e(self, K, world):
        """The same metric end to end: every layer step's q, k_new and v_new
        come in from pinned host memory, and every layer step's output goes
        back to pinned host memory, inside the model-step graphs.  Inputs come
        in eight layers per transfer (all layers in one when a model step's
        inputs total at most 1 MiB): the first chunk before the first layer
        (with seq_lens, the block table and the plan), each further chunk on a
        side stream while the chunk before it computes.  A side stream reads
        each layer's output back as soon as that layer is done.  Only the wait
        for a chunk of inputs joins the kernel chain, once per eight layers,
        so the other layers keep their programmatic dependent launch; each
        layer has its own output buffer, and the graph ends by joining the
        side streams."""
        torch, binding, LAYERS, stream = self.torch, self.binding, self.LAYERS, self.stream
        dev, q, k_new, v_new, out = self.dev, self.q, self.k_new, self.v_new, self.out
        w = self.w
        nb = lambda t: t.numel() * t.element_size()
        nq, nk = q.numel(), k_new.numel()
        per_layer = nq + 2 * nk                    # elements of one layer's inputs
        h_in = torch.empty(LAYERS * per_layer, dtype=self.elem_t).pin_memory()
        for l in range(LAYERS):                    # every layer's inputs, as the host holds them
            base = l * per_layer
            h_in[base:base + nq].copy_(q.reshape(-1).cpu())
            h_in[base + nq:base + nq + nk].copy_(k_new.reshape(-1).cpu())
            h_in[base + nq + nk:base + per_layer].copy_(v_new.reshape(-1).cpu())
        d_in = torch.empty_like(h_in, device=dev)
        hbt = torch.from_numpy(np.ascontiguousarray(w.block_table)).pin_memory()
        hsl = torch.from_numpy(np.ascontiguousarray(w.seq_lens)).pin_memory()
        hout = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(LAYERS)]
        ob = [torch.empty_like(out) for _ in range(LAYERS)]
        side_out = torch.cuda.Stream(device=dev)
        side_in = torch.cuda.Stream(device=dev)

        def layer_inputs(l):
            base = l * per_layer
            return (d_in[base:base + nq].view(q.shape),
                    d_in[base + nq:base + nq + nk].view(k_new.shape),
                    d_in[base + nq + nk:base + per_layer].view(v_new.shape))

        # layers whose inputs one transfer brings in: all of them when a model
        # step's inputs are small (one transfer, no join at all), else eight
        CHUNK = LAYERS if LAYERS * per_layer * h_in.element_size() <= (1 << 20) else 8

        def copy_in(l0, l1):
            d_in[l0 * per_layer:l1 * per_layer].copy_(h_in[l0 * per_layer:l1 * per_layer],
                                                      non_blocking=True)

        def capture_e2e(slot, nlayers):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                self.bt.copy_(hbt, non_blocking=True)
                self.sl.copy_(hsl, non_blocking=True)
                self.upload_in_graph(slot)
                copy_in(0, min(CHUNK, nlayers))
                side_out.wait_stream(stream)
                ready = {}
                for l in range(nlayers):
                    if l % CHUNK == 0:
                        nxt = l + CHUNK
                        if nxt < nlayers:  # the next chunk's inputs, while this one computes
                            side_in.wait_stream(stream)  # (fork: brings side_in into the capture)
                            with torch.cuda.stream(side_in):
                                copy_in(nxt, min(nxt + CHUNK, nlayers))
                            ready[nxt] = torch.cuda.Event()
                            ready[nxt].record(side_in)
                        if l in ready:
                            stream.wait_event(ready[l])
                    qq, kk, vv = layer_inputs(l)
                    self.layer_call(self.pools[l], qq, kk, vv, ob[l], self.ws_for(slot))
                    done = torch.cuda.Event()
                    done.record(stream)
                    side_out.wait_event(done)
                    with torch.cuda.stream(side_out):
                        hout[l].copy_(ob[l], non_blocking=True)
                if ready:  # side_in took part only if a chunk came in on it
                    stream.wait_stream(side_in)
                stream.wait_stream(side_out)
                self.join_upload()
            return g

        full, rem = divmod(K, LAYERS)
        e_full = [capture_e2e(i, LAYERS) for i in range(2)] if full else []
        e_rem = [capture_e2e(i, rem) for i in range(2)] if rem else []
        self.warm(K, e_full, e_rem)
        m0 = self.m
        e2e_ms = max_over_ranks(self.time_region(K, e_full, e_rem, world) / K, world, dev)
        nmodel = self.m - m0
        # the last layer's output, read back to the host, equals the device's
        last = rem - 1 if rem else LAYERS - 1
        if not torch.equal(hout[last].to(dev), ob[last]):
            raise RuntimeError("e2e output read back differs from the device output")
        h2d_bytes = (K * per_layer * h_in.element_size()
                     + nmodel * (nb(hbt) + nb(hsl) + int(self.plan0.c.blob_bytes)))
        return {"value": round(job_value(self.kv_bytes, e2e_ms, world), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": int(round(h2d_bytes / K)),
                "d2h_bytes_per_step": int(nb(hout[0])),
                "overlap": f"inputs come in {CHUNK} layers per transfer, each chunk while the "
                           "one before it computes; a side stream reads each layer's output "
                           "back while the next layers compute"}

    def append_us(self):
        """a1 alone: pa_kv_append as its own launch (the step fuses it into the
        split kernel), one launch per layer's cache in one graph."""
        torch, binding = self.torch, self.binding
        app_call = {"int8": binding.append_q8, "fp8": binding.append_fp8}.get(self.args.kv,
                                                                              binding.append)
        ga = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ga, stream=self.stream):
            for l in range(self.LAYERS):
                app_call(self.shape, self.k_new, self.v_new, *self.pools[l], self.bt, self.sl,
                         self.status)
        ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(self.stream):
            ga.replay()
            ev_a[0].record(self.stream)
            for _ in range(4):
                ga.replay()
            ev_a[1].record(self.stream)
        torch.cuda.synchronize()
        self.check_status()
        return ev_a[0].elapsed_time(ev_a[1]) * 1e3 / (4 * self.LAYERS)

    def workload_name(self):
        return (self.w.name + KV_NAMES.get(self.args.kv, "") +
                (", bf16" if self.args.dtype == "bf16" else ""))


REPEATS = 5   # further K-step regions, for the spread of the per-step time

# how a workload's name says which 8-bit cache it reads
KV_NAMES = {"int8": ", INT8 KV cache (per-row scales)",
            "fp8": ", FP8 (E4M3) KV cache (per-row scales)"}


def repeat_regions(db, K, gfull, grem, world, dev):
    """µs per layer step of REPEATS more K-step regions, timed exactly as
    the first (which alone gives `value`): their p10, median and p90."""
    us = sorted(max_over_ranks(db.time_region(K, gfull, grem, world) / K, world, dev) * 1e3
                for _ in range(REPEATS))
    pick = lambda q: float(np.percentile(us, q))
    return {"regions": REPEATS, "steps_each": K, "us_per_step_p10": round(pick(10), 3),
            "us_per_step_median": round(pick(50), 3), "us_per_step_p90": round(pick(90), 3)}


def run_ours(args):
    LAYERS = args.layers
    import torch

    from paged_kv_decode_24_gb300 import binding
    from paged_kv_decode_24_gb300 import build as _build

    world, rank, local = dist_setup(args)
    cpu_base = cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # before any CUDA call
        cpu_base = run_oracle_subprocess(args.config, args.cpu_seconds, args.kv, args.dtype)
        cpu_all = run_oracle_all_cores(args.config, args.cpu_seconds, args.kv, args.dtype)

    _build.ensure_built()
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    num_sms = props.multi_processor_count
    stream = torch.cuda.Stream(device=dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    peak, peak_src = read_peaks()
    K = args.steps

    db = DecodeBench(args, args.config, rank, dev, stream, num_sms, LAYERS)
    w = db.w
    graphs_full, graphs_rem = db.graphs(K)
    warm_full = graphs_full or [db.capture(i, LAYERS) for i in range(2)]
    db.warm(max(args.warmup, LAYERS), warm_full, graphs_rem or warm_full)

    uuid = None
    try:
        u = str(props.uuid)
        uuid = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass

    def sustain(seconds):
        """Untimed model steps of the same workload for about `seconds`, so the
        clock samples see the GPU under this load."""
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            db.warm(4 * LAYERS, warm_full, warm_full)

    clocks = ClockSampler(uuid)
    clocks.start()
    sustain(0.4)
    total_ms = db.time_region(K, graphs_full, graphs_rem, world)
    sustain(0.4)
    clk = clocks.stop()
    if clk is not None:
        clk["window"] = "0.4 s of the same workload before and after the timed region, and the region"
    ms_per_step = max_over_ranks(total_ms / K, world, dev)
    # the fused call is the only work in a step besides a2's amortised upload,
    # so its mean launch duration over the timed region is the step time
    dec_mean_ms = total_ms / K
    dist = repeat_regions(db, K, graphs_full, graphs_rem, world, dev)
    iso_us = db.isolated_us()
    e2e = None if args.no_e2e else db.e2e(K, world)
    append_us = db.append_us()

    achieved = db.dec_bytes / (dec_mean_ms * 1e-3) / 1e9
    value = job_value(db.kv_bytes, ms_per_step, world)
    plan0 = db.plan0
    two_kernel = args.merge == "combine"
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if args.dtype == "bf16" else "f16",
        "kv_cache": {"int8": "int8 codes + fp32 row scales",
                     "fp8": "e4m3 codes + fp32 row scales"}.get(args.kv, args.dtype),
        "accumulate": "f32",
        "data": "synthetic (seeded; shapes and value laws of the workload)",
        "config": workload_config(args, w, world),
        "run": run_dict(args, db, LAYERS, l2),
        "hbm_frac_step": round(value / world / peak, 4),
        "roofline": {
            "kernel": {"int8": "pa_append_decode_attention_q8 = split_decode_q8_kernel (INT8)",
                       "fp8": "pa_append_decode_attention_fp8 = split_decode_q8_kernel (E4M3)"}.get(
                           args.kv, "pa_append_decode_attention = split_decode_kernel") +
                      (" (with the append) + combine_kernel, timed together"
                       if two_kernel else " (with the append and the split merge)"),
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peak_src == "measured"
                           else "fallback 6800 GB/s (of fallback)",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic_for(args.config, args.kv, args.dtype, decode_family(w, args.kv)),
            "algorithmic_bytes_per_launch": db.dec_bytes,
            "us_per_launch": round(dec_mean_ms * 1e3, 3),
            "us_per_launch_isolated": round(iso_us, 3),
        },
        "distribution": dist,
        "plan_host_us": None,
        "append_us": round(append_us, 3),
        "cpu_baseline": cpu_base,
        "cpu_baseline_all_cores": cpu_all,
        "e2e": e2e,
        "gpu_launches": db.launches_per_step * K,
        "clocks": clk,
    }
    # host cost of pa_plan alone (reported, not part of the device timing)
    t0 = time.perf_counter()
    for _ in range(20):
        binding.Plan(db.shape, db.lens_host, num_sms, w.forced_splits)
    res["plan_host_us"] = round((time.perf_counter() - t0) / 20 * 1e6, 2)

    # the other workloads, timed the same way in the same run (K layer steps
    # each, after their own warm-up); reported beside the headline
    extras = [(c, kv) for c, kv in (args.also or [])
              if (c, kv or args.kv) != (args.config, args.kv)]
    if extras:
        del db, graphs_full, graphs_rem, warm_full
        torch.cuda.empty_cache()
        res["per_config"] = {}
        for c, kv in extras:
            xa = copy.copy(args)
            if kv is not None:
                xa.kv, xa.dtype = kv, "fp16"
            xb = DecodeBench(xa, c, rank, dev, stream, num_sms, LAYERS)
            gf, gr = xb.graphs(K)
            wf = gf or [xb.capture(i, LAYERS) for i in range(2)]
            xb.warm(max(args.warmup, LAYERS), wf, gr or wf)
            t_ms = xb.time_region(K, gf, gr, world)
            ms = max_over_ranks(t_ms / K, world, dev)
            xdist = repeat_regions(xb, K, gf, gr, world, dev)
            ach = xb.dec_bytes / (t_ms / K * 1e-3) / 1e9
            res["per_config"][str(c) if kv is None else f"{c}-{kv}"] = {
                "workload": xb.workload_name(),
                "us_per_step": round(ms * 1e3, 3),
                "value": round(job_value(xb.kv_bytes, ms, world), 2), "unit": "GB/s",
                "roofline_frac": round(ach / peak, 4),
                "achieved": round(ach, 1),
                "algorithmic_bytes_per_launch": xb.dec_bytes,
                "traffic": traffic_for(c, xa.kv, xa.dtype, decode_family(xb.w, xa.kv)),
                "splits": int(xb.plan0.c.max_splits),
                "gpu_launches": xb.launches_per_step * K,
                "distribution": xdist,
            }
            del xb, gf, gr, wf
            torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def workload_config(args, w, world):
    """The workload the line is about: the same dict on both arms."""
    q8 = args.kv in ("int8", "fp8")
    return {
        "workload": (w.name + KV_NAMES.get(args.kv, "") +
                     (", bf16" if args.dtype == "bf16" else "")),
        "config_id": args.config,
        "batch": w.batch,
        "heads_q_kv": f"{w.num_q_heads}/{w.num_kv_heads}",
        "head_dim": w.head_dim,
        "page_size": w.page_size,
        "sum_seq_len": int(w.seq_lens.sum()),
        "kv_read_bytes_per_step": w.kv_bytes_int8() if q8 else w.kv_bytes(),
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def run_dict(args, db, LAYERS, l2):
    """How our arm ran the workload."""
    plan0 = db.plan0
    return {
        "splits": int(plan0.c.max_splits),
        "split_merge": ("separate combine_kernel after the split kernel (plan option "
                        "merge = PA_MERGE_COMBINE_KERNEL)" if args.merge == "combine" else
                        "by the last split task of each group, inside the split kernel"),
        "work_items": int(plan0.c.num_work_items),
        "ctas": int(plan0.c.num_ctas),
        "plan_options": args.plan or "defaults",
        "early_kv": ("on: each layer's first page copies start before the wait on the layer "
                     "ahead; q and the new rows after it" if args.early_kv == "on" else "off"),
        "step": "one layer: pa_append_decode_attention (one kernel: the append fused into the "
                "split kernel, whose last split per group merges); pa_plan_upload once per "
                f"{LAYERS}-layer model step, inside the timing" +
                (" (each model step's graph uploads the next step's plan into a second "
                 "workspace while its layers run)" if args.upload == "ahead" else
                 " (before the step's first layer)") +
                "; pa_plan on the host for each model step while the GPU runs the one before it",
        "launch": f"one CUDA graph per {LAYERS}-layer model step (plan upload + the layers' "
                  "calls back to back, programmatic dependent launch between kernels); a spin "
                  "kernel before the start event keeps host launch latency out of the device "
                  "timing",
        "l2": f"{LAYERS} per-layer KV caches ({LAYERS * db.cache_bytes / 2**30:.1f} GiB) "
              f"vs {l2 / 2**20:.0f} MiB L2: each step reads pages the L2 no longer holds",
    }


# ---------------------------------------------------------------------------
# reference arm: the float64 oracle on the host cores

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    from paged_kv_decode_24_gb300 import workloads
    w = workloads.make_config(args.config, kv=args.kv, dtype=args.dtype)
    # a bounded sample per step: the whole run stays within about two minutes
    per_step = min(2.0, max(0.2, 120.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        oracle_sample(w, per_step / 4)
    total_s = 0.0
    total_kv = 0
    desc = ""
    for _ in range(args.steps):
        dt, kv, desc = oracle_sample(w, per_step)
        total_s += dt
        total_kv += kv
    value = total_kv / total_s / 1e9
    cores = 1  # BLAS threads pinned to one above; the oracle itself is single-threaded
    res = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_s / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; shapes and value laws of the workload)",
        "config": workload_config(args, w, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {desc}, about {per_step:.2f} s"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res))


# ---------------------------------------------------------------------------
# KV swap: pa_copy_blocks between the device pools and pinned host pools

SWAP_METRIC = "KV swap GB/s (pa_copy_blocks: swap-out to pinned host memory + swap-in)"


def swap_selection(w):
    """Every fourth sequence's pages, and the host slots they go to."""
    pages = []
    for b in range(0, w.batch, 4):
        n = -(-int(w.seq_lens[b]) // w.page_size)
        pages.extend(int(x) for x in w.block_table[b, :n])
    return np.array(pages, np.int32)


def run_swap(args):
    import torch

    from paged_kv_decode_24_gb300 import binding, workloads
    from paged_kv_decode_24_gb300 import build as _build

    world, rank, local = dist_setup(args)
    w = workloads.make_config(args.config, seed=workloads.SEED_BASE + args.config + 1000 * rank)
    pages = swap_selection(w)
    n = len(pages)
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        blk = np.zeros((n,) + w.k_pages.shape[1:], np.float16)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 2.0:
            pairs = np.stack([pages, np.arange(n)], 1)
            blk = oracle.copy_blocks(blk, w.k_pages, pairs)
            reps += 1
        dt = time.perf_counter() - t0
        cpu_base = {"value": round(reps * n * blk[0].nbytes / dt / 1e9, 3), "unit": "GB/s",
                    "cores": 1, "kind": "oracle",
                    "sample": f"oracle.copy_blocks of {n} K pages into a host array, "
                              f"{reps} times in {dt:.1f} s"}
    _build.ensure_built()
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    kd = torch.from_numpy(w.k_pages).to(dev)
    vd = torch.from_numpy(w.v_pages).to(dev)
    hk = torch.empty((n,) + tuple(kd.shape[1:]), dtype=kd.dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    out_pairs = torch.from_numpy(np.stack([pages, np.arange(n, dtype=np.int32)], 1)).to(dev)
    in_pairs = torch.from_numpy(np.stack([np.arange(n, dtype=np.int32), pages], 1)).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    block_bytes = kd[0].numel() * kd.element_size()
    step_bytes = 4 * n * block_bytes   # K and V, out and back in

    def step():
        binding.copy_blocks(hk, kd, out_pairs, status, stream=stream)
        binding.copy_blocks(hv, vd, out_pairs, status, stream=stream)
        binding.copy_blocks(kd, hk, in_pairs, status, stream=stream)
        binding.copy_blocks(vd, hv, in_pairs, status, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    # the link as one large copy engine transfer each way, for the peak
    big_h = torch.empty(n * block_bytes, dtype=torch.uint8).pin_memory()
    big_d = torch.empty(n * block_bytes, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            big_d.copy_(big_h, non_blocking=True)
            big_h.copy_(big_d, non_blocking=True)
        ev[0].record(stream)
        big_d.copy_(big_h, non_blocking=True)
        ev[1].record(stream)
        big_h.copy_(big_d, non_blocking=True)
        ev[2].record(stream)
    torch.cuda.synchronize()
    h2d_gbs = big_d.numel() / (ev[0].elapsed_time(ev[1]) * 1e-3) / 1e9
    d2h_gbs = big_d.numel() / (ev[1].elapsed_time(ev[2]) * 1e-3) / 1e9
    peak = 2.0 / (1.0 / h2d_gbs + 1.0 / d2h_gbs)   # the same bytes each way
    clocks = ClockSampler()
    clocks.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    K = args.steps
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(K):
            step()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x}")
    if not (torch.equal(kd.cpu(), torch.from_numpy(w.k_pages)) and
            torch.equal(vd.cpu(), torch.from_numpy(w.v_pages))):
        raise RuntimeError("pools changed across swap round trips")
    ms = max_over_ranks(start.elapsed_time(end) / K, world, dev)
    value = world * step_bytes / (ms * 1e-3) / 1e9
    res = {
        "metric": SWAP_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded; the workload's pools)",
        "config": {"workload": w.name + ": every 4th sequence swapped out and back in",
                   "config_id": args.config, "pages": n, "block_bytes": block_bytes,
                   "step": "4 pa_copy_blocks (K and V out to pinned host memory, then back)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "host link", "achieved": round(value / world, 1),
                     "peak": round(peak, 1), "unit": "GB/s", "frac": round(value / world / peak, 4),
                     "peak_source": f"measured in this run: one {n * block_bytes / 2**20:.0f} MiB "
                                    f"cudaMemcpyAsync each way ({h2d_gbs:.0f} GB/s in, "
                                    f"{d2h_gbs:.0f} GB/s out), harmonic mean",
                     "traffic": None},
        "cpu_baseline": cpu_base,
        "e2e": {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": 2 * n * block_bytes,
                "d2h_bytes_per_step": 2 * n * block_bytes,
                "note": "the step itself moves host buffers"},
        "gpu_launches": 4 * K,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# several query tokens per sequence: pa_kv_append_tokens + pa_prefill_attention

PREFILL_METRIC = "multi-token attention TFLOP/s (causal; pa_kv_append_tokens + pa_prefill_attention)"
PREFILL_LAYERS = 4


def prefill_flops(w):
    """4 D FLOPs (q.k and p.v) per query head, query token and key it sees."""
    n = 0
    for L, qn in zip(w.seq_lens.astype(np.int64), w.q_lens.astype(np.int64)):
        n += int(qn * (L - qn) + qn * (qn + 1) // 2)   # sum over queries of (position + 1)
    return 4 * w.head_dim * w.num_q_heads * n


def run_prefill(args):
    import torch

    from paged_kv_decode_24_gb300 import binding, workloads
    from paged_kv_decode_24_gb300 import build as _build

    if args.config not in (1, 2):
        raise SystemExit("--op prefill takes --config 1 or 2")
    world, rank, local = dist_setup(args)
    w = workloads.make_prefill_config(args.config, seed=workloads.SEED_BASE + 100 + args.config +
                                      1000 * rank, dtype=args.dtype)
    flops = prefill_flops(w)
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        done = 0
        rng = np.random.default_rng(0)
        while time.perf_counter() - t0 < 3.0:
            r = int(rng.integers(0, w.q.shape[0]))
            oracle.prefill_attention(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens,
                                     w.q_lens, w.scale,
                                     rows=[(r, h) for h in range(w.num_q_heads)])
            b = int(np.searchsorted(np.cumsum(w.q_lens), r, side="right"))
            pos = int(w.seq_lens[b]) - int(w.q_lens[b]) + (r - int(np.cumsum(w.q_lens)[b] - w.q_lens[b]))
            done += 4 * w.head_dim * w.num_q_heads * (pos + 1)
        dt = time.perf_counter() - t0
        cpu_base = {"value": round(done / dt / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
                    "kind": "oracle",
                    "sample": f"float64 oracle rows (all heads of random query tokens), {dt:.1f} s"}
    _build.ensure_built()
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    elem_t = torch.bfloat16 if args.dtype == "bf16" else torch.float16
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    to_elem = lambda a: to_dev(a).to(elem_t)
    shape = binding.make_shape(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size,
                               w.max_pages_per_seq, w.num_pages, args.dtype)
    q, kn, vn = to_elem(w.q), to_elem(w.k_new), to_elem(w.v_new)
    bt, sl = to_dev(w.block_table), to_dev(w.seq_lens)
    cache0 = (to_elem(w.k_pages), to_elem(w.v_pages))
    pools = [cache0] + [tuple(t.clone() for t in cache0) for _ in range(PREFILL_LAYERS - 1)]
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    plan = binding.PrefillPlan(shape, w.seq_lens, w.q_lens, rows_per_tile=args.prefill_rows)
    ws = binding.alloc_workspace(plan, dev)
    mixed = None
    if args.decode_rows == "decode-call":
        from paged_kv_decode_24_gb300.runner import MixedStep
        mixed = MixedStep(w, dev, rows_per_tile=args.prefill_rows)
        torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        binding.prefill_upload(plan, ws, stream=stream)
        if mixed is None:
            binding.append_tokens(shape, plan, kn, vn, *pools[0], bt, sl, ws, status,
                                  stream=stream)
            binding.prefill(shape, plan, q, *pools[0], bt, sl, w.scale, out, ws, status,
                            stream=stream)
        else:
            mixed.run(*pools[0], stream=stream)
    stream.synchronize()

    def layer(l):
        if mixed is None:
            binding.append_tokens(shape, plan, kn, vn, *pools[l], bt, sl, ws, status)
            binding.prefill(shape, plan, q, *pools[l], bt, sl, w.scale, out, ws, status)
        else:
            mixed.run(*pools[l], stream=stream)

    def capture(nl):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(nl):
                layer(l)
        return g

    K = args.steps
    full, rem = divmod(K, PREFILL_LAYERS)
    g_full = capture(PREFILL_LAYERS)
    g_rem = capture(rem) if rem else None
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // PREFILL_LAYERS)):
            g_full.replay()
    stream.synchronize()
    # the split of a step: attention alone, in its own events (with the
    # decode call, the whole two-stream step, appends included)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for l in range(PREFILL_LAYERS):
            if mixed is None:
                binding.prefill(shape, plan, q, *pools[l], bt, sl, w.scale, out, ws, status,
                                stream=stream)
            else:
                mixed.run(*pools[l], stream=stream)
        ev[1].record(stream)
    torch.cuda.synchronize()
    attn_ms = ev[0].elapsed_time(ev[1]) / PREFILL_LAYERS
    clocks = ClockSampler()
    clocks.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    st = int(status.item()) | (mixed.read_status() if mixed is not None else 0)
    if st != 0:
        raise RuntimeError(f"device status {st:#x}")
    ms = max_over_ranks(start.elapsed_time(end) / K, world, dev)
    value = world * flops / (ms * 1e-3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, peak_src = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        peak, peak_src = 1900.0, "fallback"
    achieved = flops / (attn_ms * 1e-3) / 1e12
    rows = int(w.q.shape[0])
    res = {
        "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if args.dtype == "bf16" else "f16",
        "data": "synthetic (seeded; shapes and value laws of the workload)",
        "config": {"workload": w.name, "config_id": args.config, "query_rows": rows,
                   "flops_per_step": flops, "tiles": int(plan.c.num_tiles),
                   "step": ("one layer: pa_kv_append_tokens + pa_prefill_attention"
                            if mixed is None else
                            f"one layer: the {len(mixed.dec)} single-token sequences through "
                            "pa_append_decode_attention on a second stream, forked from and "
                            f"joined back into the step's stream, while the other "
                            f"{len(mixed.pre)} go through pa_kv_append_tokens + "
                            "pa_prefill_attention"),
                   "launch": f"CUDA graph of {PREFILL_LAYERS} layers' calls over "
                             f"{PREFILL_LAYERS} per-layer KV caches",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": ("prefill_kernel (mma.sync m16n8k16, 64-row tiles)"
                               if args.prefill_rows == 64 else
                               "prefill_tc5_kernel (tcgen05, 128-row tiles)") +
                              ("" if mixed is None else
                               " beside split_decode_tc_kernel on a second stream: the whole "
                               "step, appends included"), "bound": "tensor",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "peak_source": "MEASURED_PEAKS.json bf16_tflops (of measured; fp16 has "
                                    "the same dense rate)" if peak_src == "measured"
                                    else "fallback 1900 TFLOP/s (of fallback)",
                     "traffic": None, "us_per_launch": round(attn_ms * 1e3, 3)},
        "cpu_baseline": cpu_base,
        "e2e": None,
        "gpu_launches": (2 if mixed is None else 3) * K,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.oracle_worker:
        oracle_worker(args)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "swap":
        run_swap(args)
    elif args.op == "prefill":
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
