"""Build libplx.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each translation unit under csrc/ compiles in parallel; the objects link into
``_build/libplx.so`` next to this file. Rebuilds only when a source or header
is newer than the library. ``python -m parametrized_local_linear_gb300.build
[--force] [--ptxas-v]``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libplx.so")
# The same sources with PLX_DEBUG_BOUNDS: device-side index checks that set
# an error bit (reported by plx_check_device_error) and skip the access
# instead of faulting. A debugging aid where no memory checker can run.
DEBUG_BUILD = os.path.join(HERE, "_build_debug")
DEBUG_LIB = os.path.join(DEBUG_BUILD, "libplx_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + [os.path.join(ROOT, "include", "plx.h"), __file__]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, ptxas_verbose: bool = False, verbose: bool = False,
          debug_bounds: bool = False) -> str:
    """Build libplx.so (or, with debug_bounds, libplx_debug.so with the
    device-side bounds checks); return its path."""
    build_dir, lib = (DEBUG_BUILD, DEBUG_LIB) if debug_bounds else (BUILD, LIB)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = nvcc_path()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                    "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    if debug_bounds:
        flags += ["-DPLX_DEBUG_BOUNDS"]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{p.stdout}\n{p.stderr}")
        return obj, p.stdout + p.stderr

    with ThreadPoolExecutor(max_workers=len(_sources())) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose or ptxas_verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, ptxas_verbose="--ptxas-v" in sys.argv, verbose=True,
                debug_bounds="--debug-bounds" in sys.argv))
