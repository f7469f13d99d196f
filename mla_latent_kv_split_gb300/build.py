"""Builds ``libmla_decode.so`` in-tree with nvcc for sm_103a (no cmake, no torch).

Each ``csrc/*.cu`` is compiled to an object in parallel, then linked into one shared
library under ``mla_latent_kv_split_gb300/lib/``.  Rebuilds only when a source or header
is newer than the library.
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
LIBDIR = os.path.join(PKG, "lib")
BUILDDIR = os.path.join(PKG, "_build")
LIB = os.path.join(LIBDIR, "libmla_decode.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmla_decode.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [
        os.path.join(ROOT, "include", "mla_decode.h"), os.path.abspath(__file__)]


# A test build of the same sources (never loaded by the package): every bounded wait gives
# up after 20 ms instead of 4 s (and a waiting warp sleeps at most 0.1 ms at a time), and the exported mla_fault_injection_drop_tile makes one
# CTA leave one tile unloaded, so that tests can run the kernel's abort path.
FAULT_LIB = os.path.join(LIBDIR, "libmla_decode_fault_injection.so")
FAULT_FLAGS = ("-DMLA_FAULT_INJECTION", "-DMLA_WAIT_LIMIT_NS=20000000ull")


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def flags(extra=()):
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                   "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr", *extra]


def build(verbose: bool = False, force: bool = False, extra=(), fault_injection: bool = False) -> str:
    lib = FAULT_LIB if fault_injection else LIB
    builddir = BUILDDIR + ("_fault_injection" if fault_injection else "")
    if fault_injection:
        extra = (*extra, *FAULT_FLAGS)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(LIBDIR, exist_ok=True)
    os.makedirs(builddir, exist_ok=True)
    cc = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(builddir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *flags(extra), "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, flush=True)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv,
                extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ()))
