"""Build libgdnspec.so in-tree for sm_103a (GB300).

    python -m speculative_decode_hybrid_gb300.build [--force] [--verbose] [--debug]

Each .cu / .cpp translation unit is compiled in parallel with nvcc (one
-gencode: arch=compute_103a, code=sm_103a) into _build/, then linked into
speculative_decode_hybrid_gb300/_lib/libgdnspec.so against the shared CUDA
runtime. No cmake; a full rebuild takes well under a minute.

--debug builds the bounds-checking variant instead (_build_debug/ ->
_lib/libgdnspec_debug.so, compiled with GDN_DEBUG_BOUNDS): every global
access of every kernel is checked against its buffer's extent, and an access
that would fall outside is skipped and flagged GDN_DEV_BOUNDS in the call's
dev_status word (no trap). Load it with gdnspec.load(path) or the
GDNSPEC_LIB environment variable; the release library is untouched.
"""
from __future__ import annotations

import argparse
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
BUILD = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libgdnspec.so")
BUILD_DEBUG = os.path.join(ROOT, "_build_debug")
LIB_DEBUG = os.path.join(LIBDIR, "libgdnspec_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdnspec")
    return cand


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(lib: str = None) -> bool:
    lib = lib or LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, verbose: bool, ptxas_v: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD_DEBUG if debug else BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + (["-DGDN_DEBUG_BOUNDS"] if debug else []) + ["-c", src, "-o", obj]
    if ptxas_v and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if ptxas_v:
        sys.stdout.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False, debug: bool = False) -> str:
    """Compile and link the library (debug=True: the bounds-checking variant); returns its path."""
    lib = LIB_DEBUG if debug else LIB
    if not force and not ptxas_v and up_to_date(lib):
        return lib
    os.makedirs(BUILD_DEBUG if debug else BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, ptxas_v, debug), srcs))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-v", action="store_true", help="print registers / spills / smem per kernel")
    ap.add_argument("--debug", action="store_true", help="the bounds-checking variant (libgdnspec_debug.so)")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, ptxas_v=a.ptxas_v, debug=a.debug))
