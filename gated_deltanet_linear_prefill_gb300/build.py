"""Builds libgdn.so (the C-ABI library) in-tree for sm_103a with nvcc.

Every translation unit under csrc/ is compiled in parallel into an object,
then linked into one shared library with the CUDA runtime linked statically
and no other dependency (the driver entry points the tensor-core kernel needs
are fetched at run time). Run as a module or call build().

Two more libraries come from the same sources for diagnosis only (nothing loads
them by default): build(trace=True) makes libgdn_trace.so with -DGDN_TC_TRACE (the
chunk kernel records per-role clock stamps, include/gdn_trace.h), and
build(checked=True) makes libgdn_checked.so with -DGDN_CHECKED (every global index
the kernels compute from their inputs is checked against its buffer; a failure
reports GDN_ERR_BOUNDS and skips the access).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libgdn.so")
TRACE_LIB = os.path.join(HERE, "libgdn_trace.so")
CHECKED_LIB = os.path.join(HERE, "libgdn_checked.so")
BUILD_DIR = os.path.join(HERE, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "gdn.h"),
                                                               os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, trace: bool = False, checked: bool = False) -> str:
    if trace and checked:
        raise ValueError("one diagnostic build at a time")
    lib = TRACE_LIB if trace else CHECKED_LIB if checked else LIB
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    bdir = os.path.join(BUILD_DIR, "trace" if trace else "checked") if (trace or checked) else BUILD_DIR
    os.makedirs(bdir, exist_ok=True)
    objs = []
    extra = ["-DGDN_TC_TRACE"] if trace else ["-DGDN_CHECKED"] if checked else []

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc] + ARCH + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, len(sources()))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
