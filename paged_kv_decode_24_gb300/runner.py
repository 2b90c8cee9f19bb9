"""Device-side holder for one decode step's buffers, driving the C ABI.

Moves a host workload into torch CUDA tensors once, then issues
pa_kv_append / pa_plan / pa_plan_upload / pa_decode_attention (and their
8-bit-cache forms, INT8 or FP8, when the workload carries one) through ``binding``.  It
holds no arithmetic of its own.
"""

from __future__ import annotations

import numpy as np

from . import binding


class DeviceDecode:
    def __init__(self, w, device="cuda", num_sms=None):
        import torch
        self.torch = torch
        self.w = w
        self.device = torch.device(device)
        elem = torch.bfloat16 if getattr(w, "dtype", "fp16") == "bf16" else None

        def t(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(self.device)

        def te(a):
            # element arrays; bf16 workloads hold bf16-exact float32 values, so
            # the cast is exact
            x = t(a)
            return x.to(elem) if elem is not None else x

        self.q = te(w.q)
        self.k_new = te(w.k_new)
        self.v_new = te(w.v_new)
        self.k_pages = te(w.k_pages)
        self.v_pages = te(w.v_pages)
        self.block_table = t(w.block_table)
        self.seq_lens = t(w.seq_lens)
        self.q8 = w.k_codes is not None   # the workload also carries an 8-bit cache
        self.kv = w.kv                    # its format: "int8" or "fp8"
        if self.q8:
            self.k_codes = t(w.k_codes)
            self.v_codes = t(w.v_codes)
            self.k_scales = t(w.k_scales)
            self.v_scales = t(w.v_scales)
        self.out = torch.empty_like(self.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.shape = binding.shape_of(self.q, self.k_pages, self.block_table)
        self.shape.batch = len(w.seq_lens)   # q may hold several rows per sequence
        if num_sms is None:
            num_sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        self.num_sms = int(num_sms)
        self.plan_obj = None
        self.workspace = None

    def make_plan(self, forced_splits=None, seq_lens_host=None, **options):
        """pa_plan (or pa_plan_ex when plan options are named, e.g.
        merge="combine", wait_limit_ns=...) and its upload."""
        fs = self.w.forced_splits if forced_splits is None else forced_splits
        lens = self.w.seq_lens if seq_lens_host is None else seq_lens_host
        opts = binding.plan_options(**options) if options else None
        self.plan_obj = binding.Plan(self.shape, lens, self.num_sms, fs, options=opts)
        need = self.plan_obj.workspace_bytes
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = binding.alloc_workspace(self.plan_obj, self.device)
        binding.upload(self.plan_obj, self.workspace)
        return self.plan_obj

    def append(self):
        binding.append(self.shape, self.k_new, self.v_new, self.k_pages, self.v_pages,
                       self.block_table, self.seq_lens, self.status)

    def decode(self, out=None):
        if self.plan_obj is None:
            self.make_plan()
        binding.decode(self.shape, self.plan_obj, self.q, self.k_pages, self.v_pages,
                       self.block_table, self.seq_lens, self.w.scale,
                       self.out if out is None else out, self.workspace, self.status)
        return self.out if out is None else out

    def append_decode(self, out=None):
        """pa_append_decode_attention: the step's append and attention in one launch."""
        if self.plan_obj is None:
            self.make_plan()
        dst = self.out if out is None else out
        binding.append_decode(self.shape, self.plan_obj, self.q, self.k_new, self.v_new,
                              self.k_pages, self.v_pages, self.block_table, self.seq_lens,
                              self.w.scale, dst, self.workspace, self.status)
        return dst

    def append_q8(self):
        binding.append_q8(self.shape, self.k_new, self.v_new, self.k_codes, self.v_codes,
                          self.k_scales, self.v_scales, self.block_table, self.seq_lens,
                          self.status)

    def decode_q8(self, out=None):
        if self.plan_obj is None:
            self.make_plan()
        dst = self.out if out is None else out
        binding.decode_q8(self.shape, self.plan_obj, self.q, self.k_codes, self.v_codes,
                          self.k_scales, self.v_scales, self.block_table, self.seq_lens,
                          self.w.scale, dst, self.workspace, self.status)
        return dst

    def append_decode_q8(self, out=None):
        if self.plan_obj is None:
            self.make_plan()
        dst = self.out if out is None else out
        binding.append_decode_q8(self.shape, self.plan_obj, self.q, self.k_new, self.v_new,
                                 self.k_codes, self.v_codes, self.k_scales, self.v_scales,
                                 self.block_table, self.seq_lens, self.w.scale, dst,
                                 self.workspace, self.status)
        return dst

    def append_fp8(self):
        binding.append_fp8(self.shape, self.k_new, self.v_new, self.k_codes, self.v_codes,
                           self.k_scales, self.v_scales, self.block_table, self.seq_lens,
                           self.status)

    def decode_fp8(self, out=None):
        if self.plan_obj is None:
            self.make_plan()
        dst = self.out if out is None else out
        binding.decode_fp8(self.shape, self.plan_obj, self.q, self.k_codes, self.v_codes,
                           self.k_scales, self.v_scales, self.block_table, self.seq_lens,
                           self.w.scale, dst, self.workspace, self.status)
        return dst

    def append_decode_fp8(self, out=None):
        if self.plan_obj is None:
            self.make_plan()
        dst = self.out if out is None else out
        binding.append_decode_fp8(self.shape, self.plan_obj, self.q, self.k_new, self.v_new,
                                  self.k_codes, self.v_codes, self.k_scales, self.v_scales,
                                  self.block_table, self.seq_lens, self.w.scale, dst,
                                  self.workspace, self.status)
        return dst

    # the 8-bit cache the workload carries (INT8 or FP8)
    def append8(self):
        return self.append_fp8() if self.kv == "fp8" else self.append_q8()

    def decode8(self, out=None):
        return self.decode_fp8(out) if self.kv == "fp8" else self.decode_q8(out)

    def append_decode8(self, out=None):
        return self.append_decode_fp8(out) if self.kv == "fp8" else self.append_decode_q8(out)

    # ---- several query tokens per sequence (workloads made with q_lens)

    def make_prefill_plan(self, seq_lens_host=None, rows_per_tile=0, wait_limit_ns=0):
        lens = self.w.seq_lens if seq_lens_host is None else seq_lens_host
        self.pf_plan = binding.PrefillPlan(self.shape, lens, self.w.q_lens,
                                           rows_per_tile=rows_per_tile,
                                           wait_limit_ns=wait_limit_ns)
        self.pf_ws = binding.alloc_workspace(self.pf_plan, self.device)
        binding.prefill_upload(self.pf_plan, self.pf_ws)
        return self.pf_plan

    def append_tokens(self):
        binding.append_tokens(self.shape, self.pf_plan, self.k_new, self.v_new, self.k_pages,
                              self.v_pages, self.block_table, self.seq_lens, self.pf_ws,
                              self.status)

    def prefill(self, out=None):
        dst = self.out if out is None else out
        binding.prefill(self.shape, self.pf_plan, self.q, self.k_pages, self.v_pages,
                        self.block_table, self.seq_lens, self.w.scale, dst, self.pf_ws,
                        self.status)
        return dst

    def gather_slots(self):
        width = self.shape.max_pages_per_seq * self.shape.page_size
        slots = self.torch.empty((self.shape.batch, width), dtype=self.torch.int32,
                                 device=self.device)
        binding.gather_indices(self.shape, self.block_table, self.seq_lens, slots, self.status)
        return slots

    def read_status(self) -> int:
        self.torch.cuda.synchronize(self.device)
        return int(self.status.item())


class MixedStep:
    """A multi-token step whose batch mixes prefill chunks with single-token
    decodes (swiftLLM's piggybacked prefill and decode), served on two
    streams as an engine would serve it: the sequences with one query token
    through pa_append_decode_attention, the others through
    pa_kv_append_tokens + pa_prefill_attention.  Both parts read and write
    the same pools through their own rows of the block table (their pages
    are distinct).  The second stream forks from the caller's stream and
    joins back into it, so the step is ordered like one call.  This class
    only selects rows on the host and issues the calls.

    The decode part is planned as if it had a third of the SMs
    (decode_sms): its plan then cuts fewer splits, so fewer decode CTAs, and
    the tile CTAs of the other part find shared memory beside them on every
    SM, so the two parts run at once instead of in turn."""

    def __init__(self, w, device="cuda", num_sms=None, rows_per_tile=0, decode_sms=None):
        import torch
        self.torch = torch
        self.w = w
        self.device = torch.device(device)
        elem = torch.bfloat16 if getattr(w, "dtype", "fp16") == "bf16" else torch.float16
        ql = np.asarray(w.q_lens, np.int64)
        cu = np.concatenate([[0], np.cumsum(ql)])
        self.dec = np.nonzero(ql == 1)[0]
        self.pre = np.nonzero(ql != 1)[0]
        self.rows_dec = cu[self.dec]
        self.rows_pre = (np.concatenate([np.arange(cu[b], cu[b + 1]) for b in self.pre])
                         if len(self.pre) else np.zeros(0, np.int64)).astype(np.int64)

        def t(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(self.device)

        def te(a):
            return t(a).to(elem)

        dtype = getattr(w, "dtype", "fp16")
        if num_sms is None:
            num_sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        S, mp = w.page_size, w.max_pages_per_seq
        # decode part
        self.shape_d = binding.make_shape(len(self.dec), w.num_q_heads, w.num_kv_heads,
                                          w.head_dim, S, mp, w.num_pages, dtype)
        self.q_d = te(w.q[self.rows_dec])
        self.kn_d, self.vn_d = te(w.k_new[self.rows_dec]), te(w.v_new[self.rows_dec])
        self.bt_d, self.sl_d = t(w.block_table[self.dec]), t(w.seq_lens[self.dec])
        self.out_d = torch.empty_like(self.q_d)
        self.status_d = torch.zeros(1, dtype=torch.int32, device=self.device)
        if decode_sms is None:
            decode_sms = max(1, int(num_sms) // 3)
        self.plan_d = self.ws_d = None
        if len(self.dec):   # an empty part makes no plan and launches nothing
            self.plan_d = binding.Plan(self.shape_d, np.ascontiguousarray(w.seq_lens[self.dec]),
                                       int(decode_sms))
            self.ws_d = binding.alloc_workspace(self.plan_d, self.device)
            binding.upload(self.plan_d, self.ws_d)
        # prefill part
        self.shape_p = binding.make_shape(len(self.pre), w.num_q_heads, w.num_kv_heads,
                                          w.head_dim, S, mp, w.num_pages, dtype)
        self.q_p = te(w.q[self.rows_pre])
        self.kn_p, self.vn_p = te(w.k_new[self.rows_pre]), te(w.v_new[self.rows_pre])
        self.bt_p, self.sl_p = t(w.block_table[self.pre]), t(w.seq_lens[self.pre])
        self.out_p = torch.empty_like(self.q_p)
        self.status_p = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.plan_p = self.ws_p = None
        if len(self.pre):
            self.plan_p = binding.PrefillPlan(self.shape_p,
                                              np.ascontiguousarray(w.seq_lens[self.pre]),
                                              np.ascontiguousarray(w.q_lens[self.pre]),
                                              rows_per_tile=rows_per_tile)
            self.ws_p = binding.alloc_workspace(self.plan_p, self.device)
            binding.prefill_upload(self.plan_p, self.ws_p)
        self.side = torch.cuda.Stream(device=self.device)
        self.ev_fork = torch.cuda.Event()
        self.ev_join = torch.cuda.Event()

    def run(self, k_pages, v_pages, stream=None):
        """The step over pools (k_pages, v_pages) on `stream` (default: the
        current stream), the decode part on a second stream in between."""
        torch = self.torch
        s0 = torch.cuda.current_stream(self.device) if stream is None else stream
        self.ev_fork.record(s0)
        self.side.wait_event(self.ev_fork)
        if len(self.dec):
            binding.append_decode(self.shape_d, self.plan_d, self.q_d, self.kn_d, self.vn_d,
                                  k_pages, v_pages, self.bt_d, self.sl_d, self.w.scale,
                                  self.out_d, self.ws_d, self.status_d, stream=self.side)
        if len(self.pre):
            binding.append_tokens(self.shape_p, self.plan_p, self.kn_p, self.vn_p, k_pages,
                                  v_pages, self.bt_p, self.sl_p, self.ws_p, self.status_p,
                                  stream=s0)
            binding.prefill(self.shape_p, self.plan_p, self.q_p, k_pages, v_pages, self.bt_p,
                            self.sl_p, self.w.scale, self.out_p, self.ws_p, self.status_p,
                            stream=s0)
        self.ev_join.record(self.side)
        s0.wait_event(self.ev_join)

    def output(self):
        """Every query row's output, in the batch's row order."""
        torch = self.torch
        out = torch.empty((self.w.q.shape[0], self.w.num_q_heads, self.w.head_dim),
                          dtype=self.q_d.dtype, device=self.device)
        out[torch.from_numpy(self.rows_dec).to(self.device)] = self.out_d
        out[torch.from_numpy(self.rows_pre).to(self.device)] = self.out_p
        return out

    def read_status(self) -> int:
        self.torch.cuda.synchronize(self.device)
        return int(self.status_d.item()) | int(self.status_p.item())
