"""Build libkda_gb300.so from csrc/*.cu with nvcc for sm_103a (in-tree, no cmake).

Each translation unit is compiled in parallel, then linked into one shared library under
``_build/<machine>/``.  A rebuild happens when any source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build", platform.machine())
LIB_PATH = os.path.join(BUILD_DIR, "libkda_gb300.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkda_gb300")
    return path


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


# The debug variant (-DKDA_DEBUG: device-side bounds checks in the tensor-core prefill), built on
# demand into a directory of its own; the release library is the one the package loads.
DEBUG_BUILD_DIR = BUILD_DIR + "-debug"
DEBUG_LIB_PATH = os.path.join(DEBUG_BUILD_DIR, "libkda_gb300_debug.so")


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    """Compile and link the library (or, with debug=True, its bounds-checked variant); returns its
    path."""
    lib_path, build_dir = (DEBUG_LIB_PATH, DEBUG_BUILD_DIR) if debug else (LIB_PATH, BUILD_DIR)
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + ARCH_FLAGS + list(extra_flags or []) + ["-I", INCLUDE] + (["-DKDA_DEBUG"] if debug else [])
    if verbose:
        flags = flags + ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, "-c", src, "-o", obj] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=min(8, len(sources()))) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose:
        for _, log in results:
            if log:
                print(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    # -ldl: the NVTX ranges of the C ABI look up a profiler's injection library at run time
    cmd = [cc, "-shared", "-o", tmp] + [o for o, _ in results] + ARCH_FLAGS + ["-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
