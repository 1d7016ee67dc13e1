"""Build libinkling_rel_attn.so in-tree with nvcc for sm_103a.

The translation units are compiled in parallel; the shared library links the
CUDA runtime statically and resolves the driver's tensor-map encoder through
the runtime at run time, so it needs no libcuda at link time.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libinkling_rel_attn.so")
SOURCES = ["api.cu", "decode.cu", "decode_noalloc.cu", "prefill.cu", "selftest.cu", "kv_append.cu",
           "kv_conv.cu"]
HEADERS = ["ptx.cuh", "internal.h", "tc.cuh", "plan.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
         "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_dep() -> float:
    paths = [os.path.join(CSRC, h) for h in HEADERS] + [
        os.path.join(ROOT, "include", "inkling_rel_attn.h")]
    return max((os.path.getmtime(p) for p in paths if os.path.exists(p)), default=0.0)


def _compile(src: str, extra, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    srcp = os.path.join(CSRC, src)
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(srcp), _newest_dep()):
        return obj
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", srcp, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        print(r.stderr, file=sys.stderr)
    return obj


def build(verbose: bool = False, extra_flags=None) -> str:
    """Compile every translation unit and link the shared library; returns
    its path.  Up-to-date objects are reused."""
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra_flags or [])
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose), SOURCES))
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
