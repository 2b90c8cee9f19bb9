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
