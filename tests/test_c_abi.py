"""The C ABI from plain C: include/pagedattn.h compiles as C99 with warnings
as errors, and a C program linked against libpagedattn.so exercises the
host-only entry points (plans, the block allocator, the multi-token plan),
with no GPU and no Python in between; it also reports the public structs'
layout, which the ctypes binding must match.
"""

from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_and_host_calls_from_c(lib, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from paged_kv_decode_24_gb300 import binding
    libdir = os.path.dirname(binding.LIB_PATH)
    exe = str(tmp_path / "abi_host")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c", "abi_host.c"), "-o", exe,
                        "-L", libdir, "-lpagedattn", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi ok" in r.stdout
    _check_layouts(r.stdout)


def _check_layouts(report):
    """The ctypes structures of the binding have the C structs' sizes and
    field offsets, as the C compiler lays them out."""
    from paged_kv_decode_24_gb300 import binding
    classes = {"pa_shape_t": binding.PaShape, "pa_plan_t": binding.PaPlan,
               "pa_plan_options_t": binding.PaPlanOptions,
               "pa_prefill_plan_t": binding.PaPrefillPlan,
               "pa_prefill_options_t": binding.PaPrefillOptions}
    seen = set()
    for line in report.splitlines():
        if not line.startswith("layout "):
            continue
        words = line.split()
        name, size, pairs = words[1], int(words[2]), words[3:]
        cls = classes[name]
        assert ctypes.sizeof(cls) == size, (name, ctypes.sizeof(cls), size)
        for field, off in zip(pairs[::2], pairs[1::2]):
            assert getattr(cls, field).offset == int(off), (name, field)
        seen.add(name)
    assert seen == set(classes)


@pytest.mark.gpu
def test_decode_from_c_on_gpu(lib, tmp_path):
    """pa_kv_append -> pa_plan -> pa_plan_upload -> pa_decode_attention, then
    pa_append_decode_attention_fp8, from a C program: one token per sequence,
    so each head's output is exactly the new V row of its KV head."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    from paged_kv_decode_24_gb300 import binding
    libdir = os.path.dirname(binding.LIB_PATH)
    exe = str(tmp_path / "abi_gpu")
    r = subprocess.run([nvcc, "-x", "c", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c", "abi_gpu.c"), "-o", exe,
                        "-L", libdir, "-lpagedattn", "-Xlinker", "-rpath=" + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "decode from C ok" in r.stdout
