"""Build libw4a16.so in-tree with nvcc for sm_103a.

Every .cu file is compiled to an object in parallel, then the objects are
linked into the shared library. The debug flavor, libw4a16_debug.so, is the
same sources with -DW4A16_DEBUG_CHECKS: the decode stream's index checks
record the first failure in a device word (w4a16_debug_check_word) and skip
the access instead of touching memory out of range.

Usage: python -m weight_only_bit_04_b300.build [--force] [--verbose] [--debug | --all]
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libw4a16.so")
OBJ_DIR = os.path.join(HERE, "_build")
LIB_DEBUG = os.path.join(HERE, "libw4a16_debug.so")
OBJ_DIR_DEBUG = os.path.join(HERE, "_build_debug")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libw4a16.so")
    return cand


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in sources() + _headers())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib, obj_dir = (LIB_DEBUG, OBJ_DIR_DEBUG) if debug else (LIB, OBJ_DIR)
    defines = ["-DW4A16_DEBUG_CHECKS"] if debug else []
    if not force and not _stale(lib):
        return lib
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    newest_header = max(os.path.getmtime(p) for p in _headers())

    def compile_one(src: str):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        if (not force and os.path.exists(obj) and os.path.getmtime(obj) > os.path.getmtime(src)
                and os.path.getmtime(obj) > newest_header):
            return obj, None
        cmd = [cc, *ARCH, *FLAGS, *defines, "-I", INCLUDE, "-c", src, "-o", obj + ".tmp"]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(obj + ".tmp", obj)
        return obj, r

    with ThreadPoolExecutor(max_workers=max(1, min(len(sources()), os.cpu_count() or 1))) as pool:
        results = list(pool.map(compile_one, sources()))
    failed = False
    for obj, r in results:
        if r is None:
            continue
        if verbose or r.returncode != 0:
            sys.stdout.write(r.stdout)
            sys.stderr.write(r.stderr)
        failed |= r.returncode != 0
    name = os.path.basename(lib)
    if failed:
        raise RuntimeError(f"nvcc failed building {name}")
    cmd = [cc, *ARCH, "--shared", "-o", lib + ".tmp", *[obj for obj, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stderr)
        raise RuntimeError(f"nvcc failed linking {name}")
    os.replace(lib + ".tmp", lib)
    return lib


def build_all(force: bool = False, verbose: bool = False) -> list[str]:
    """The release library and its debug flavor."""
    return [build(force, verbose), build(force, verbose, debug=True)]


if __name__ == "__main__":
    force, verbose = "--force" in sys.argv, "--verbose" in sys.argv
    if "--all" in sys.argv:
        print("\n".join(build_all(force, verbose)))
    else:
        print(build(force, verbose, debug="--debug" in sys.argv))
