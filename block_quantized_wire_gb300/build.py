"""Build libbq.so (the CUDA library behind the C ABI in include/bq.h) for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into a shared
library next to this file. Arithmetic flags: no fused multiply-add contraction
(``--fmad=false``), IEEE division and square root, no flush-to-zero, so the kernels'
results are fixed by their explicit ``__f*_rn`` operations alone.
"""
from __future__ import annotations

import concurrent.futures
import fcntl
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libbq.so")
OBJDIR = os.path.join(PKG, "_build")
# The same sources with the compile-time alternatives of the measured defaults: the
# 8-value-per-lane quantize, accumulate and ring hop, the bulk-copy-staged hops, no
# 256-bit accesses. Tests build it to keep those paths bit-exact too.
ALT_LIB = os.path.join(PKG, "libbq_alt.so")
ALT_OBJDIR = os.path.join(PKG, "_build_alt")
ALT_FLAGS = ["-DBQ_ACCUM_WIDE=0", "-DBQ_QUANT_WIDE=0", "-DBQ_HOP_WIDE=0", "-DBQ_MX_WIDE=0", "-DBQ_WIDE_V8=0"]
# The same sources with the loading and CTA-size choices that the per-lane async copies
# and the one-CTA-per-SM launches were measured against: direct loads in the accumulates
# and the fused reduce, 256-thread CTAs everywhere. Tests build it to keep those paths
# bit-exact too.
DIRECT_LIB = os.path.join(PKG, "libbq_direct.so")
DIRECT_OBJDIR = os.path.join(PKG, "_build_direct")
DIRECT_FLAGS = ["-DBQ_ACCUM_ASYNC=0", "-DBQ_ACCUM_MX_ASYNC=0", "-DBQ_REDUCE_ASYNC=0", "-DBQ_QUANT_WIDE_THREADS=256",
                "-DBQ_HOP_WIDE_THREADS=256", "-DBQ_QUANT_E4M3_THREADS=256", "-DBQ_DEQUANT_MX_THREADS=256"]
# The debug build: every kernel checks each global access against the buffers its
# arguments describe and counts (instead of performing) an access outside them.
DEBUG_LIB = os.path.join(PKG, "libbq_debug.so")
DEBUG_OBJDIR = os.path.join(PKG, "_build_debug")
DEBUG_FLAGS = ["-DBQ_DEBUG=1"]

SOURCES = ["bq_api.cu", "bq_i8.cu", "bq_mx.cu", "bq_mx_wire.cu", "bq_e4m3.cu"]
HEADERS = ["bq_device.cuh", "bq_launch.h", "bq_chunks.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3", "-std=c++17", "-lineinfo", "--fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbq.so")


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "bq.h"), __file__]
    return files


def _stamp_path(lib: str) -> str:
    return lib + ".flags"


def _flag_stamp(extra_flags) -> str:
    return "\n".join([*ARCH, *NVCC_FLAGS, *extra_flags]) + "\n"


def up_to_date(lib: str = LIB, extra_flags=()) -> bool:
    """True if `lib` is newer than every source and was built with exactly these flags
    (recorded in the stamp file written next to it by the build)."""
    if not os.path.exists(lib):
        return False
    try:
        with open(_stamp_path(lib)) as f:
            if f.read() != _flag_stamp(extra_flags):
                return False
    except OSError:
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build_library(force: bool = False, verbose: bool = False, extra_flags=(), lib: str = LIB,
                  objdir: str = OBJDIR) -> str:
    """Compile and link `lib` (libbq.so) if any source is newer than it; returns its path.

    Concurrent callers (one process per GPU under torchrun) are serialized by a file
    lock: the first builds, the others find the library up to date. The library is
    replaced atomically, so a process that already loaded it is unaffected."""
    if not force and up_to_date(lib, extra_flags):
        return lib
    os.makedirs(objdir, exist_ok=True)
    with open(os.path.join(objdir, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and up_to_date(lib, extra_flags):
                return lib
            return _build_locked(verbose, extra_flags, lib, objdir)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def build_alt_library(force: bool = False, verbose: bool = False) -> str:
    """Build libbq_alt.so: the sources with ALT_FLAGS."""
    return build_library(force, verbose, ALT_FLAGS, ALT_LIB, ALT_OBJDIR)


def build_direct_library(force: bool = False, verbose: bool = False) -> str:
    """Build libbq_direct.so: the sources with DIRECT_FLAGS."""
    return build_library(force, verbose, DIRECT_FLAGS, DIRECT_LIB, DIRECT_OBJDIR)


def build_debug_library(force: bool = False, verbose: bool = False) -> str:
    """Build libbq_debug.so: the sources with DEBUG_FLAGS."""
    return build_library(force, verbose, DEBUG_FLAGS, DEBUG_LIB, DEBUG_OBJDIR)


def _build_locked(verbose: bool, extra_flags, lib: str, objdir: str) -> str:
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-I", CSRC, "-c",
               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".%d.tmp" % os.getpid()
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(_stamp_path(lib) + ".tmp", "w") as f:
        f.write(_flag_stamp(extra_flags))
    os.replace(_stamp_path(lib) + ".tmp", _stamp_path(lib))
    return lib


if __name__ == "__main__":
    # Extra flags build the default library with them; its stamp then records them, so
    # the next default build (tests, bench) sees the mismatch and rebuilds.
    flags = sys.argv[1:]
    print(build_library(force=True, verbose=True, extra_flags=flags))
