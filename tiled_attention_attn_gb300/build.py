"""Builds libattn.so in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel into ``_build/`` and linked into
``tiled_attention_attn_gb300/libattn.so``; a rebuild happens only when a
source or header is newer than the library.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build", "attn")
LIB_PATH = os.path.join(PKG, "libattn.so")
TRACE_LIB_PATH = os.path.join(PKG, "libattn_trace.so")   # phase-trace points compiled in

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["attn_host.cu", "attn_noalloc.cu", "attn_pad.cu", "attn_rotary.cu", "attn_bwd.cu", "attn_bwd_d64.cu",
           "attn_bwd_d128.cu", "attn_kernels_d64.cu", "attn_kernels_d128.cu", "attn_plan.cpp", "attn_decode.cu",
           "attn_pair_d128.cu", "attn_decode_tc.cu", "attn_kernels_rope.cu", "attn_kernels_sorted.cu"]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe is None and os.path.exists("/usr/local/cuda/bin/nvcc"):
        exe = "/usr/local/cuda/bin/nvcc"
    if exe is None:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")
    return exe


def _deps():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files += glob.glob(os.path.join(CSRC, "*.inc")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return files


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    """Build libattn.so, or with ``trace`` the phase-traced libattn_trace.so."""
    out = TRACE_LIB_PATH if trace else LIB_PATH
    if not force and up_to_date(out):
        return out
    bdir = BUILD_DIR + ("_trace" if trace else "")
    os.makedirs(bdir, exist_ok=True)
    exe = nvcc()
    common = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if trace:
        common += ["-DATTN_TRACE=1"]

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
        cmd = [exe, "-c", os.path.join(CSRC, src), "-o", obj] + common + ARCH
        if src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"] if verbose else []
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + ".tmp"
    cmd = [exe, "-shared", "-o", tmp] + objs + ARCH
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, trace="--trace" in sys.argv))
