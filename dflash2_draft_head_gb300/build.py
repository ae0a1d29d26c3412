"""Build libdflash2.so in-tree with nvcc for sm_103a (GB300).

Each .cu file under csrc/ is compiled in parallel into _build/, then linked
into dflash2_draft_head_gb300/libdflash2.so (static CUDA runtime).  The build
is skipped when the library is newer than every source and header.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdflash2.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-Wall,-Wextra",
              "-Werror", "all-warnings", f"-I{INCLUDE}"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdflash2.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(INCLUDE, "dflash2.h"), os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", *ARCH, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


TRACE_LIB = os.path.join(PKG, "libdflash2_trace.so")


TRACED = ("select.cu", "topk.cu")


def build_traced(force: bool = False) -> str:
    """The library with the phase traces compiled in (the selector's and the
    streaming top-K's sources with -DDF2_TRACE, every other object from the
    normal build): a separate libdflash2_trace.so for measurement; the normal
    library is unchanged."""
    build()
    deps = _deps() + [LIB]
    if not force and os.path.exists(TRACE_LIB) and \
            all(os.path.getmtime(p) <= os.path.getmtime(TRACE_LIB) for p in deps):
        return TRACE_LIB
    nvcc = _nvcc()
    tdir = os.path.join(BUILD, "trace")
    os.makedirs(tdir, exist_ok=True)

    def compile_one(name):
        obj = os.path.join(tdir, name[:-3] + ".o")
        r = subprocess.run([nvcc, *NVCC_FLAGS, "-DDF2_TRACE", "-c", os.path.join(CSRC, name),
                            "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name} (traced):\n{r.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(TRACED)) as ex:
        list(ex.map(compile_one, TRACED))
    objs = [os.path.join(tdir if os.path.basename(src) in TRACED else BUILD,
                         os.path.basename(src)[:-3] + ".o") for src in _sources()]
    tmp = TRACE_LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, "-shared", *ARCH, "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed (traced):\n{r.stderr}")
    os.replace(tmp, TRACE_LIB)
    return TRACE_LIB


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv, verbose=True))
