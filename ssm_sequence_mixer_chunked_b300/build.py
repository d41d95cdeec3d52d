"""Build libtm2.so in-tree with nvcc for sm_103a (B300).

    python -m ssm_sequence_mixer_chunked_b300.build [--force] [--verbose] [--debug]

Each .cu under csrc/ is compiled to an object in _build/ (in parallel), then linked
into ssm_sequence_mixer_chunked_b300/libtm2.so with a static CUDA runtime.  The
library is rebuilt only when a source or header is newer than it.  --debug builds the
bounds-checked variant, libtm2_debug.so (objects in _build/debug, -DTM2_DEBUG): device-side
index checks that record TM2_ERR_BOUNDS in the status word instead of accessing, and a
stream synchronisation plus status check after every launch (the binding loads it when the
environment sets TM2_DEBUG=1).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtm2.so")
LIB_DEBUG = os.path.join(PKG, "libtm2_debug.so")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC]
# Approximate exp / divide / reciprocal only where the arithmetic is bf16-bound anyway (the
# tensor-core kernels, whose parity bar is 2e-2).  The fp32 path (CUDA-core kernels, decode,
# the A-mask running sums shared by every path) keeps IEEE division and the accurate library
# functions, so its 1e-4 bar does not rest on approximations.
FAST_MATH_PREFIX = "tm2_tc"


def _flags(src: str):
    fast = os.path.basename(src).startswith(FAST_MATH_PREFIX)
    return CFLAGS + (["--use_fast_math"] if fast else [])


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(OBJDIR, "debug" if debug else "", os.path.basename(src)[:-3] + ".o")
    cmd = [NVCC, *ARCH, *_flags(src), *(["-DTM2_DEBUG"] if debug else []), "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    if not force and up_to_date(lib):
        return lib
    os.makedirs(os.path.join(OBJDIR, "debug") if debug else OBJDIR, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), srcs))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [NVCC, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv, debug="--debug" in sys.argv))
