"""Build libpagedattn.so in-tree with nvcc for sm_103a.

Each source is compiled in parallel to an object under ``_build/`` and
linked into ``paged_kv_decode_24_gb300/_lib/libpagedattn.so`` with the CUDA
runtime linked statically, so the library loads without a GPU.  The build is
skipped when the library is newer than every source and header.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libpagedattn.so")

SOURCES = ["api.cu", "plan.cpp", "aux_kernels.cu", "decode_d64.cu", "decode_d128.cu",
           "decode_tc_d64.cu", "decode_tc_d128.cu", "decode_q8_d64.cu", "decode_q8_d128.cu",
           "decode_f8_d64.cu", "decode_f8_d128.cu",
           "static_workspace.cu", "blocks.cpp", "prefill_plan.cpp", "prefill_d64.cu",
           "prefill_d128.cu", "prefill_tc5_d64.cu", "prefill_tc5_d128.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedattn")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "pagedattn.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj, *ARCH, *COMMON]
    if src.endswith(".cpp"):
        cmd = [nvcc(), "-c", "-x", "c++", os.path.join(CSRC, src), "-o", obj, *COMMON]
    elif verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build_library(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile and link libpagedattn.so; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc(), "-shared", *ARCH, "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def ensure_built() -> str:
    return build_library(force=False)


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
