"""ctypes binding of libpagedattn (include/pagedattn.h).

Argument marshalling only.  Torch tensors supply device memory and the
current CUDA stream; every computation runs in the library's kernels.  There
is no fallback: if the shared library is missing or a call fails, this module
raises.
"""

from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libpagedattn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "pagedattn.h")

PA_DEV_BAD_PAGE = 0x1
PA_DEV_BAD_SEQ_LEN = 0x2
PA_DEV_PLAN_MISMATCH = 0x4
PA_DEV_TIMEOUT = 0x8

STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_WORKSPACE",
                4: "PA_ERR_CUDA", 5: "PA_ERR_DEVICE_OOB", 6: "PA_ERR_TIMEOUT",
                7: "PA_ERR_NO_MEMORY", 8: "PA_ERR_PLAN"}


class PaShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("dtype", ctypes.c_int32)]


PA_DTYPE_F16 = 0
PA_DTYPE_BF16 = 1
DTYPES = {"fp16": PA_DTYPE_F16, "bf16": PA_DTYPE_BF16}


class PaPlan(ctypes.Structure):
    _fields_ = [("shape", PaShape), ("num_work_items", ctypes.c_int32),
                ("num_groups", ctypes.c_int32), ("num_split_items", ctypes.c_int32),
                ("max_splits", ctypes.c_int32), ("chunk_pages", ctypes.c_int32),
                ("num_ctas", ctypes.c_int32), ("num_shared_ctas", ctypes.c_int32),
                ("warps_per_cta", ctypes.c_int32),
                ("owns_blob", ctypes.c_int32), ("plan_id", ctypes.c_uint64),
                ("blob_bytes", ctypes.c_size_t), ("workspace_bytes", ctypes.c_size_t),
                ("host_blob", ctypes.c_void_p), ("merge", ctypes.c_int32),
                ("l2_prefetch_pages", ctypes.c_int32), ("l2_prefetch_ctas", ctypes.c_int32),
                ("q8_stages", ctypes.c_int32), ("wait_limit_ns", ctypes.c_uint64),
                ("early_kv", ctypes.c_int32)]


PA_MERGE_IN_SPLIT_KERNEL = 0
PA_MERGE_COMBINE_KERNEL = 1
MERGES = {"split": PA_MERGE_IN_SPLIT_KERNEL, "combine": PA_MERGE_COMBINE_KERNEL}


class PaPlanOptions(ctypes.Structure):
    _fields_ = [("min_chunk_pages", ctypes.c_int32), ("waves", ctypes.c_int32),
                ("bundle_max_pages", ctypes.c_int32), ("bundle_waves", ctypes.c_int32),
                ("merge", ctypes.c_int32), ("l2_prefetch_pages", ctypes.c_int32),
                ("l2_prefetch_ctas", ctypes.c_int32), ("q8_stages", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_uint64), ("early_kv", ctypes.c_int32)]


class PaPrefillPlan(ctypes.Structure):
    _fields_ = [("shape", PaShape), ("num_tiles", ctypes.c_int32), ("total_q", ctypes.c_int32),
                ("owns_blob", ctypes.c_int32), ("rows_per_tile", ctypes.c_int32),
                ("plan_id", ctypes.c_uint64), ("blob_bytes", ctypes.c_size_t),
                ("workspace_bytes", ctypes.c_size_t), ("host_blob", ctypes.c_void_p),
                ("wait_limit_ns", ctypes.c_uint64)]


class PaPrefillOptions(ctypes.Structure):
    _fields_ = [("rows_per_tile", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_uint64)]


def plan_options(**kw) -> PaPlanOptions:
    """pa_plan_options_t from keyword fields (merge may be "split" or "combine");
    unnamed fields stay 0, their default."""
    o = PaPlanOptions()
    for k, v in kw.items():
        if k == "merge" and isinstance(v, str):
            v = MERGES[v]
        if not hasattr(o, k):
            raise TypeError(f"unknown plan option {k}")
        setattr(o, k, int(v))
    return o


class PagedAttnError(RuntimeError):
    def __init__(self, fn, code, lib):
        self.code = code
        msg = lib.pa_status_string(code).decode() if lib is not None else "?"
        super().__init__(f"{fn} returned {STATUS_NAMES.get(code, code)}: {msg}")


_lib = None

_P = ctypes.c_void_p
_SIGS = {
    "pa_kv_append": (ctypes.c_int, [ctypes.POINTER(PaShape), _P, _P, _P, _P, _P, _P, _P, _P]),
    "pa_plan": (ctypes.c_int, [ctypes.POINTER(PaShape), _P, ctypes.c_int32, ctypes.c_int32,
                               ctypes.POINTER(PaPlan)]),
    "pa_plan_in": (ctypes.c_int, [ctypes.POINTER(PaShape), _P, ctypes.c_int32, ctypes.c_int32, _P,
                                  ctypes.c_size_t, ctypes.POINTER(PaPlan)]),
    "pa_plan_ex": (ctypes.c_int, [ctypes.POINTER(PaShape), _P, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.POINTER(PaPlanOptions), _P, ctypes.c_size_t,
                                  ctypes.POINTER(PaPlan)]),
    "pa_plan_free": (None, [ctypes.POINTER(PaPlan)]),
    "pa_plan_upload": (ctypes.c_int, [ctypes.POINTER(PaPlan), _P, ctypes.c_size_t, _P]),
    "pa_decode_attention": (ctypes.c_int, [ctypes.POINTER(PaShape), ctypes.POINTER(PaPlan), _P, _P,
                                           _P, _P, _P, ctypes.c_float, _P, _P, ctypes.c_size_t,
                                           _P, _P]),
    "pa_append_decode_attention": (ctypes.c_int, [ctypes.POINTER(PaShape), ctypes.POINTER(PaPlan),
                                                  _P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P,
                                                  _P, ctypes.c_size_t, _P, _P]),
    "pa_decode_attention_static": (ctypes.c_int, [ctypes.POINTER(PaShape), ctypes.POINTER(PaPlan),
                                                  _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P]),
    "pa_kv_append_q8": (ctypes.c_int, [ctypes.POINTER(PaShape), _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P]),
    "pa_decode_attention_q8": (ctypes.c_int, [ctypes.POINTER(PaShape), ctypes.POINTER(PaPlan), _P,
                                              _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                              ctypes.c_size_t, _P, _P]),
    "pa_append_decode_attention_q8": (ctypes.c_int, [ctypes.POINTER(PaShape),
                                                     ctypes.POINTER(PaPlan), _P, _P, _P, _P, _P,
                                                     _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                                     ctypes.c_size_t, _P, _P]),
    "pa_kv_append_fp8": (ctypes.c_int, [ctypes.POINTER(PaShape), _P, _P, _P, _P, _P, _P, _P, _P,
                                        _P, _P]),
    "pa_decode_attention_fp8": (ctypes.c_int, [ctypes.POINTER(PaShape), ctypes.POINTER(PaPlan),
                                               _P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                               ctypes.c_size_t, _P, _P]),
    "pa_append_decode_attention_fp8": (ctypes.c_int, [ctypes.POINTER(PaShape),
                                                      ctypes.POINTER(PaPlan), _P, _P, _P, _P, _P,
                                                      _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                                      ctypes.c_size_t, _P, _P]),
    "pa_profile_num_blocks": (ctypes.c_int64, [ctypes.POINTER(PaShape), ctypes.c_int32,
                                               ctypes.c_int32, ctypes.c_size_t, ctypes.c_size_t]),
    "pa_block_allocator_create": (ctypes.c_int, [ctypes.c_int32, ctypes.POINTER(_P)]),
    "pa_block_allocator_destroy": (None, [_P]),
    "pa_block_num_free": (ctypes.c_int32, [_P]),
    "pa_block_alloc": (ctypes.c_int, [_P, ctypes.c_int32, _P]),
    "pa_block_free": (ctypes.c_int, [_P, _P, ctypes.c_int32]),
    "pa_block_table_grow": (ctypes.c_int, [_P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32]),
    "pa_copy_blocks": (ctypes.c_int, [_P, ctypes.c_int32, _P, ctypes.c_int32, ctypes.c_size_t, _P,
                                      ctypes.c_int32, _P, _P]),
    "pa_prefill_plan": (ctypes.c_int, [ctypes.POINTER(PaShape), _P, _P,
                                       ctypes.POINTER(PaPrefillPlan)]),
    "pa_prefill_plan_ex": (ctypes.c_int, [ctypes.POINTER(PaShape), _P, _P,
                                          ctypes.POINTER(PaPrefillOptions),
                                          ctypes.POINTER(PaPrefillPlan)]),
    "pa_prefill_plan_free": (None, [ctypes.POINTER(PaPrefillPlan)]),
    "pa_prefill_plan_upload": (ctypes.c_int, [ctypes.POINTER(PaPrefillPlan), _P, ctypes.c_size_t,
                                              _P]),
    "pa_kv_append_tokens": (ctypes.c_int, [ctypes.POINTER(PaShape), ctypes.POINTER(PaPrefillPlan),
                                           _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "pa_prefill_attention": (ctypes.c_int, [ctypes.POINTER(PaShape),
                                            ctypes.POINTER(PaPrefillPlan), _P, _P, _P, _P, _P,
                                            ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P]),
    "pa_debug_gather_indices": (ctypes.c_int, [ctypes.POINTER(PaShape), _P, _P, _P, _P, _P]),
    "pa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pa_version": (ctypes.c_char_p, []),
}


def declared_functions(header: str = HEADER) -> list[str]:
    """Names of the functions include/pagedattn.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def load(path: str = LIB_PATH):
    """Load the shared library (once) and attach signatures.  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libpagedattn not built ({path} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, code: int):
    if code != 0:
        raise PagedAttnError(fn, code, _lib)


def make_shape(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages_per_seq,
               num_pages, dtype="fp16") -> PaShape:
    """pa_shape_t; dtype "fp16" or "bf16" (or the PA_DTYPE_* code)."""
    code = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    return PaShape(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size),
                   int(max_pages_per_seq), int(num_pages), code)


class Plan:
    """Owner of a pa_plan_t; frees the host task list when collected.

    With ``host_buffer`` (a host tensor or numpy array, e.g. pinned memory)
    the task list is written there by pa_plan_in instead of a malloc'ed block.
    With ``options`` (a PaPlanOptions, see plan_options) the plan is made by
    pa_plan_ex.
    """

    def __init__(self, shape: PaShape, seq_lens_host, num_sms: int, forced_splits: int = 0,
                 host_buffer=None, options: PaPlanOptions | None = None):
        lib = load()
        self.shape = shape
        self.c = PaPlan()
        lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
        self._lens = lens
        lp = lens.ctypes.data if lens.size else None
        ptr, nbytes = None, 0
        if host_buffer is not None:
            self._buf = host_buffer
            ptr, nbytes = _host_ptr(host_buffer)
        if options is not None:
            self.options = options
            code = lib.pa_plan_ex(ctypes.byref(shape), lp, int(num_sms), int(forced_splits),
                                  ctypes.byref(options), ptr, nbytes, ctypes.byref(self.c))
        elif host_buffer is None:
            code = lib.pa_plan(ctypes.byref(shape), lp, int(num_sms), int(forced_splits),
                               ctypes.byref(self.c))
        else:
            code = lib.pa_plan_in(ctypes.byref(shape), lp, int(num_sms), int(forced_splits), ptr,
                                  nbytes, ctypes.byref(self.c))
        _check("pa_plan", code)

    def structure(self):
        c = self.c
        return (c.num_work_items, c.num_groups, c.num_split_items, c.num_ctas, c.blob_bytes)

    @property
    def workspace_bytes(self) -> int:
        return int(self.c.workspace_bytes)

    def blob(self) -> np.ndarray:
        """The task list as int32 (host copy, for inspection and tests)."""
        n = int(self.c.blob_bytes) // 4
        buf = (ctypes.c_int32 * n).from_address(self.c.host_blob)
        return np.frombuffer(buf, dtype=np.int32, count=n).copy()

    def free(self):
        if _lib is not None and getattr(self, "c", None) is not None and self.c.host_blob:
            _lib.pa_plan_free(ctypes.byref(self.c))

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def _host_ptr(buf):
    """(address, bytes) of a host numpy array or CPU torch tensor."""
    if isinstance(buf, np.ndarray):
        if not buf.flags["C_CONTIGUOUS"]:
            raise ValueError("host buffer must be contiguous")
        return ctypes.c_void_p(buf.ctypes.data), buf.nbytes
    if getattr(buf, "is_cuda", True) or not buf.is_contiguous():
        raise ValueError("host buffer must be a contiguous CPU tensor or numpy array")
    return ctypes.c_void_p(buf.data_ptr()), buf.numel() * buf.element_size()


# --------------------------------------------------------------------------
# torch-facing wrappers

def _torch():
    import torch
    return torch


def _dev_ptr(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def shape_of(q, k_pages, block_table) -> PaShape:
    torch = _torch()
    B, Hq, D = q.shape
    P, Hkv, S, D2 = k_pages.shape
    if D2 != D:
        raise ValueError("head_dim of q and k_pages differ")
    dtype = "bf16" if q.dtype == torch.bfloat16 else "fp16"
    return make_shape(B, Hq, Hkv, D, S, block_table.shape[1], P, dtype)


def _elem(shape):
    """The torch element type of q, the pools, the new rows and out for this shape."""
    torch = _torch()
    return torch.bfloat16 if shape.dtype == PA_DTYPE_BF16 else torch.float16


def append(shape, k_new, v_new, k_pages, v_pages, block_table, seq_lens, status, stream=None):
    torch = _torch()
    lib = load()
    et = _elem(shape)
    _check("pa_kv_append", lib.pa_kv_append(
        ctypes.byref(shape), _dev_ptr(k_new, et, "k_new"),
        _dev_ptr(v_new, et, "v_new"), _dev_ptr(k_pages, et, "k_pages"),
        _dev_ptr(v_pages, et, "v_pages"), _dev_ptr(block_table, torch.int32, "block_table"),
        _dev_ptr(seq_lens, torch.int32, "seq_lens"), _dev_ptr(status, torch.int32, "status"),
        _stream(stream)))


def upload(plan: Plan, workspace, stream=None):
    torch = _torch()
    lib = load()
    _check("pa_plan_upload", lib.pa_plan_upload(
        ctypes.byref(plan.c), _dev_ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)))


def decode(shape, plan: Plan, q, k_pages, v_pages, block_table, seq_lens, scale, out, workspace,
           status, stream=None):
    torch = _torch()
    lib = load()
    et = _elem(shape)
    _check("pa_decode_attention", lib.pa_decode_attention(
        ctypes.byref(shape), ctypes.byref(plan.c), _dev_ptr(q, et, "q"),
        _dev_ptr(k_pages, et, "k_pages"), _dev_ptr(v_pages, et, "v_pages"),
        _dev_ptr(block_table, torch.int32, "block_table"), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
        ctypes.c_float(scale), _dev_ptr(out, et, "out"),
        _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


def append_decode(shape, plan: Plan, q, k_new, v_new, k_pages, v_pages, block_table, seq_lens,
                  scale, out, workspace, status, stream=None):
    """pa_append_decode_attention: append the new token and attend, one launch."""
    torch = _torch()
    lib = load()
    et = _elem(shape)
    _check("pa_append_decode_attention", lib.pa_append_decode_attention(
        ctypes.byref(shape), ctypes.byref(plan.c), _dev_ptr(q, et, "q"),
        _dev_ptr(k_new, et, "k_new"), _dev_ptr(v_new, et, "v_new"),
        _dev_ptr(k_pages, et, "k_pages"), _dev_ptr(v_pages, et, "v_pages"),
        _dev_ptr(block_table, torch.int32, "block_table"), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
        ctypes.c_float(scale), _dev_ptr(out, et, "out"),
        _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


def _q8_pools(k_codes, v_codes, k_scales, v_scales, code_dtype=None):
    torch = _torch()
    cd = torch.int8 if code_dtype is None else code_dtype
    return (_dev_ptr(k_codes, cd, "k_codes"), _dev_ptr(v_codes, cd, "v_codes"),
            _dev_ptr(k_scales, torch.float32, "k_scales"),
            _dev_ptr(v_scales, torch.float32, "v_scales"))


def append_q8(shape, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens,
              status, stream=None):
    """pa_kv_append_q8: quantise the new rows into the INT8 cache."""
    torch = _torch()
    lib = load()
    _check("pa_kv_append_q8", lib.pa_kv_append_q8(
        ctypes.byref(shape), _dev_ptr(k_new, torch.float16, "k_new"),
        _dev_ptr(v_new, torch.float16, "v_new"), *_q8_pools(k_codes, v_codes, k_scales, v_scales),
        _dev_ptr(block_table, torch.int32, "block_table"), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


def decode_q8(shape, plan: Plan, q, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens,
              scale, out, workspace, status, stream=None):
    """pa_decode_attention_q8: decode over the INT8 cache."""
    torch = _torch()
    lib = load()
    _check("pa_decode_attention_q8", lib.pa_decode_attention_q8(
        ctypes.byref(shape), ctypes.byref(plan.c), _dev_ptr(q, torch.float16, "q"),
        *_q8_pools(k_codes, v_codes, k_scales, v_scales),
        _dev_ptr(block_table, torch.int32, "block_table"), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
        ctypes.c_float(scale), _dev_ptr(out, torch.float16, "out"),
        _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


def append_decode_q8(shape, plan: Plan, q, k_new, v_new, k_codes, v_codes, k_scales, v_scales,
                     block_table, seq_lens, scale, out, workspace, status, stream=None):
    """pa_append_decode_attention_q8: append the new token and attend, one launch."""
    torch = _torch()
    lib = load()
    _check("pa_append_decode_attention_q8", lib.pa_append_decode_attention_q8(
        ctypes.byref(shape), ctypes.byref(plan.c), _dev_ptr(q, torch.float16, "q"),
        _dev_ptr(k_new, torch.float16, "k_new"), _dev_ptr(v_new, torch.float16, "v_new"),
        *_q8_pools(k_codes, v_codes, k_scales, v_scales),
        _dev_ptr(block_table, torch.int32, "block_table"), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
        ctypes.c_float(scale), _dev_ptr(out, torch.float16, "out"),
        _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


def append_fp8(shape, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens,
               status, stream=None):
    """pa_kv_append_fp8: quantise the new rows into the FP8 (E4M3) cache."""
    torch = _torch()
    lib = load()
    _check("pa_kv_append_fp8", lib.pa_kv_append_fp8(
        ctypes.byref(shape), _dev_ptr(k_new, torch.float16, "k_new"),
        _dev_ptr(v_new, torch.float16, "v_new"),
        *_q8_pools(k_codes, v_codes, k_scales, v_scales, torch.uint8),
        _dev_ptr(block_table, torch.int32, "block_table"), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


def decode_fp8(shape, plan: Plan, q, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens,
               scale, out, workspace, status, stream=None):
    """pa_decode_attention_fp8: decode over the FP8 (E4M3) cache."""
    torch = _torch()
    lib = load()
    _check("pa_decode_attention_fp8", lib.pa_decode_attention_fp8(
        ctypes.byref(shape), ctypes.byref(plan.c), _dev_ptr(q, torch.float16, "q"),
        *_q8_pools(k_codes, v_codes, k_scales, v_scales, torch.uint8),
        _dev_ptr(block_table, torch.int32, "block_table"), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
        ctypes.c_float(scale), _dev_ptr(out, torch.float16, "out"),
        _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


def append_decode_fp8(shape, plan: Plan, q, k_new, v_new, k_codes, v_codes, k_scales, v_scales,
                      block_table, seq_lens, scale, out, workspace, status, stream=None):
    """pa_append_decode_attention_fp8: append the new token and attend, one launch."""
    torch = _torch()
    lib = load()
    _check("pa_append_decode_attention_fp8", lib.pa_append_decode_attention_fp8(
        ctypes.byref(shape), ctypes.byref(plan.c), _dev_ptr(q, torch.float16, "q"),
        _dev_ptr(k_new, torch.float16, "k_new"), _dev_ptr(v_new, torch.float16, "v_new"),
        *_q8_pools(k_codes, v_codes, k_scales, v_scales, torch.uint8),
        _dev_ptr(block_table, torch.int32, "block_table"), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
        ctypes.c_float(scale), _dev_ptr(out, torch.float16, "out"),
        _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


STATIC_WORKSPACE_BYTES = 16 << 20   # PA_STATIC_WORKSPACE_BYTES


def decode_static(shape, plan: Plan, q, k_pages, v_pages, block_table, seq_lens, scale, out,
                  status, stream=None):
    """pa_decode_attention_static: decode with the library's own scratch array."""
    torch = _torch()
    lib = load()
    et = _elem(shape)
    _check("pa_decode_attention_static", lib.pa_decode_attention_static(
        ctypes.byref(shape), ctypes.byref(plan.c), _dev_ptr(q, et, "q"),
        _dev_ptr(k_pages, et, "k_pages"), _dev_ptr(v_pages, et, "v_pages"),
        _dev_ptr(block_table, torch.int32, "block_table"), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
        ctypes.c_float(scale), _dev_ptr(out, et, "out"),
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


def gather_indices(shape, block_table, seq_lens, out_slots, status, stream=None):
    torch = _torch()
    lib = load()
    _check("pa_debug_gather_indices", lib.pa_debug_gather_indices(
        ctypes.byref(shape), _dev_ptr(block_table, torch.int32, "block_table"),
        _dev_ptr(seq_lens, torch.int32, "seq_lens"), _dev_ptr(out_slots, torch.int32, "out_slots"),
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


# --------------------------------------------------------------------------
# several query tokens per sequence

class PrefillPlan:
    """Owner of a pa_prefill_plan_t (tile list and row offsets, host side)."""

    def __init__(self, shape: PaShape, seq_lens_host, q_lens_host, rows_per_tile: int = 0,
                 wait_limit_ns: int = 0):
        lib = load()
        self.shape = shape
        self.c = PaPrefillPlan()
        self._lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
        self._qlens = np.ascontiguousarray(np.asarray(q_lens_host, dtype=np.int32))
        lp = self._lens.ctypes.data if self._lens.size else None
        qp = self._qlens.ctypes.data if self._qlens.size else None
        if rows_per_tile or wait_limit_ns:
            self.options = PaPrefillOptions(int(rows_per_tile), 0, int(wait_limit_ns))
            code = lib.pa_prefill_plan_ex(ctypes.byref(shape), lp, qp,
                                          ctypes.byref(self.options), ctypes.byref(self.c))
        else:
            code = lib.pa_prefill_plan(ctypes.byref(shape), lp, qp, ctypes.byref(self.c))
        _check("pa_prefill_plan", code)

    @property
    def workspace_bytes(self) -> int:
        return int(self.c.workspace_bytes)

    def blob(self) -> np.ndarray:
        n = int(self.c.blob_bytes) // 4
        buf = (ctypes.c_int32 * n).from_address(self.c.host_blob)
        return np.frombuffer(buf, dtype=np.int32, count=n).copy()

    def free(self):
        if _lib is not None and getattr(self, "c", None) is not None and self.c.host_blob:
            _lib.pa_prefill_plan_free(ctypes.byref(self.c))

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def prefill_upload(plan: PrefillPlan, workspace, stream=None):
    torch = _torch()
    _check("pa_prefill_plan_upload", load().pa_prefill_plan_upload(
        ctypes.byref(plan.c), _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)))


def append_tokens(shape, plan: PrefillPlan, k_new, v_new, k_pages, v_pages, block_table,
                  seq_lens, workspace, status, stream=None):
    """pa_kv_append_tokens: the step's new rows into their pages."""
    torch = _torch()
    et = _elem(shape)
    _check("pa_kv_append_tokens", load().pa_kv_append_tokens(
        ctypes.byref(shape), ctypes.byref(plan.c), _dev_ptr(k_new, et, "k_new"),
        _dev_ptr(v_new, et, "v_new"), _dev_ptr(k_pages, et, "k_pages"),
        _dev_ptr(v_pages, et, "v_pages"), _dev_ptr(block_table, torch.int32, "block_table"),
        _dev_ptr(seq_lens, torch.int32, "seq_lens"), _dev_ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), _dev_ptr(status, torch.int32, "status"), _stream(stream)))


def prefill(shape, plan: PrefillPlan, q, k_pages, v_pages, block_table, seq_lens, scale, out,
            workspace, status, stream=None):
    """pa_prefill_attention: every query row of the plan."""
    torch = _torch()
    et = _elem(shape)
    _check("pa_prefill_attention", load().pa_prefill_attention(
        ctypes.byref(shape), ctypes.byref(plan.c), _dev_ptr(q, et, "q"),
        _dev_ptr(k_pages, et, "k_pages"), _dev_ptr(v_pages, et, "v_pages"),
        _dev_ptr(block_table, torch.int32, "block_table"), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
        ctypes.c_float(scale), _dev_ptr(out, et, "out"), _dev_ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), _dev_ptr(status, torch.int32, "status"), _stream(stream)))


# --------------------------------------------------------------------------
# KV blocks: page counts, the free list, block copies

PA_KV_16BIT = 0
PA_KV_INT8 = 1
PA_KV_FP8 = 2


def profile_num_blocks(shape, num_layers, kv_kind, free_bytes, reserve_bytes=0) -> int:
    """pa_profile_num_blocks: pages of num_layers layers' K and V that fit."""
    n = load().pa_profile_num_blocks(ctypes.byref(shape), int(num_layers), int(kv_kind),
                                     int(free_bytes), int(reserve_bytes))
    if n < 0:
        raise PagedAttnError("pa_profile_num_blocks", 1, _lib)
    return int(n)


class BlockAllocator:
    """Owner of a pa_block_allocator_t (host free list of pages)."""

    def __init__(self, num_blocks: int):
        lib = load()
        self._h = ctypes.c_void_p()
        _check("pa_block_allocator_create",
               lib.pa_block_allocator_create(int(num_blocks), ctypes.byref(self._h)))

    def num_free(self) -> int:
        return int(load().pa_block_num_free(self._h))

    def alloc(self, n: int) -> np.ndarray:
        out = np.empty(max(int(n), 0), np.int32)
        _check("pa_block_alloc", load().pa_block_alloc(self._h, int(n),
                                                       out.ctypes.data if n else None))
        return out

    def free(self, blocks):
        b = np.ascontiguousarray(np.asarray(blocks, np.int32))
        _check("pa_block_free", load().pa_block_free(self._h, b.ctypes.data if b.size else None,
                                                     int(b.size)))

    def grow(self, row: np.ndarray, page_size: int, old_len: int, new_len: int):
        """pa_block_table_grow on a contiguous int32 numpy row, in place."""
        if row.dtype != np.int32 or not row.flags["C_CONTIGUOUS"]:
            raise ValueError("row must be a contiguous int32 array")
        _check("pa_block_table_grow", load().pa_block_table_grow(
            self._h, row.ctypes.data, int(row.size), int(page_size), int(old_len), int(new_len)))

    def close(self):
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.pa_block_allocator_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _pool_ptr(t, name):
    """A pool for pa_copy_blocks: a CUDA tensor or a pinned host tensor."""
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous torch tensor")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be on a CUDA device or in pinned host memory")
    return ctypes.c_void_p(t.data_ptr())


def copy_blocks(dst_pool, src_pool, pairs, status, stream=None):
    """pa_copy_blocks: dst_pool[d] = src_pool[s] for every (s, d) row of the
    device int32 [n, 2] tensor pairs.  Pools are [blocks, ...] tensors of the
    same block shape and dtype, on the device or in pinned host memory."""
    torch = _torch()
    if dst_pool.dtype != src_pool.dtype or tuple(dst_pool.shape[1:]) != tuple(src_pool.shape[1:]):
        raise ValueError("pools differ in block shape or dtype")
    block_bytes = int(np.prod(dst_pool.shape[1:])) * dst_pool.element_size()
    n = int(pairs.shape[0])
    _check("pa_copy_blocks", load().pa_copy_blocks(
        _pool_ptr(dst_pool, "dst_pool"), int(dst_pool.shape[0]), _pool_ptr(src_pool, "src_pool"),
        int(src_pool.shape[0]), block_bytes, _dev_ptr(pairs, torch.int32, "pairs"), n,
        _dev_ptr(status, torch.int32, "status"), _stream(stream)))


def alloc_workspace(plan: Plan, device="cuda"):
    """A uint8 device buffer of the plan's workspace size (256-byte aligned by torch)."""
    torch = _torch()
    return torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)


class Prepared:
    """A library call with its ctypes arguments converted once.

    Calling it re-issues the same call (same buffers, same stream) with no
    per-call Python marshalling; used where host overhead would otherwise
    dominate a short kernel.  The tensors are kept alive by the object.
    """

    def __init__(self, name, args, keep):
        self._fn = getattr(load(), name)
        self._name = name
        self._args = tuple(args)
        self._keep = keep

    def __call__(self):
        code = self._fn(*self._args)
        if code != 0:
            raise PagedAttnError(self._name, code, _lib)


def prepare_append(shape, k_new, v_new, k_pages, v_pages, block_table, seq_lens, status,
                   stream=None) -> Prepared:
    torch = _torch()
    et = _elem(shape)
    args = [ctypes.byref(shape), _dev_ptr(k_new, et, "k_new"),
            _dev_ptr(v_new, et, "v_new"), _dev_ptr(k_pages, et, "k_pages"),
            _dev_ptr(v_pages, et, "v_pages"),
            _dev_ptr(block_table, torch.int32, "block_table"),
            _dev_ptr(seq_lens, torch.int32, "seq_lens"), _dev_ptr(status, torch.int32, "status"),
            _stream(stream)]
    return Prepared("pa_kv_append", args, (shape, k_new, v_new, k_pages, v_pages, block_table,
                                           seq_lens, status))


def prepare_decode(shape, plan: Plan, q, k_pages, v_pages, block_table, seq_lens, scale, out,
                   workspace, status, stream=None) -> Prepared:
    torch = _torch()
    et = _elem(shape)
    args = [ctypes.byref(shape), ctypes.byref(plan.c), _dev_ptr(q, et, "q"),
            _dev_ptr(k_pages, et, "k_pages"), _dev_ptr(v_pages, et, "v_pages"),
            _dev_ptr(block_table, torch.int32, "block_table"),
            _dev_ptr(seq_lens, torch.int32, "seq_lens"), ctypes.c_float(scale),
            _dev_ptr(out, et, "out"), _dev_ptr(workspace, torch.uint8, "workspace"),
            ctypes.c_size_t(workspace.numel()), _dev_ptr(status, torch.int32, "status"),
            _stream(stream)]
    return Prepared("pa_decode_attention", args, (shape, plan, q, k_pages, v_pages, block_table,
                                                  seq_lens, out, workspace, status))


def prepare_upload(plan: Plan, workspace, stream=None) -> Prepared:
    torch = _torch()
    args = [ctypes.byref(plan.c), _dev_ptr(workspace, torch.uint8, "workspace"),
            ctypes.c_size_t(workspace.numel()), _stream(stream)]
    return Prepared("pa_plan_upload", args, (plan, workspace))
