"""Build ``librope_gb300.so`` in-tree with nvcc for sm_103a.

Usage: ``python -m transformer_rope_positional_gb300.build [--force] [--verbose] [--debug]``.
The translation units compile in parallel; the shared library lands in
``transformer_rope_positional_gb300/lib/``.  The CUDA runtime is linked
statically, so the library needs only the driver at run time.

``--debug`` builds ``librope_gb300_debug.so`` with ``-DROPE_DEBUG_BOUNDS``:
every global access of every kernel is checked against the span of the tensor
it addresses; an access outside it is skipped and recorded in the device error
word (ROPE_DEVICE_INDEX_OUT_OF_BOUNDS).  The binding loads it instead of the
release library when ``ROPE_GB300_DEBUG_BOUNDS=1`` is set.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import fcntl
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "lib")
LIB_PATH = os.path.join(LIB_DIR, "librope_gb300.so")
DEBUG_LIB_PATH = os.path.join(LIB_DIR, "librope_gb300_debug.so")

SOURCES = ["rope_api.cu", "rope_launch.cu", "rope_inplace_fwd.cu", "rope_inplace_bwd.cu", "rope_cache.cu",
           "rope_qkv.cu"]
HEADERS = ["rope_device.cuh", "rope_launch.h", "rope_inplace.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or add CUDA's bin directory to PATH)")


def _inputs():
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    return srcs + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "rope_gb300.h")]


def up_to_date(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile every translation unit and link the shared library (the
    bounds-checking debug library with ``debug=True``).  Processes that build
    at once (one per rank of a multi-GPU run) take turns on a lock file: the
    object files share one build directory."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(LIB_DIR, exist_ok=True)
    with open(lib_path + ".lock", "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and up_to_date(lib_path):  # built while this process waited
                return lib_path
            return _build_locked(lib_path, verbose, debug)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(lib_path: str, verbose: bool, debug: bool) -> str:
    build_dir = BUILD_DIR + ("_debug" if debug else "")
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if verbose else []) + (["-DROPE_DEBUG_BOUNDS"] if debug else [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib_path + ".%d.tmp" % os.getpid()
    cmd = [cc, *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/spill reports")
    ap.add_argument("--debug", action="store_true", help="the bounds-checking debug library")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose, debug=args.debug))
