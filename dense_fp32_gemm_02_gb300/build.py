"""Build libsgemm.so in-tree with nvcc for sm_103a (no torch extension machinery):
the translation units under csrc/ compile in parallel, then one link.

``python -m dense_fp32_gemm_02_gb300.build`` or ``build()`` from Python.
The library is written to ``dense_fp32_gemm_02_gb300/_build/libsgemm.so``;
a build is skipped when the library is newer than every source file.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libsgemm.so")
# the range-checked build (-DSGEMM_DEBUG_BOUNDS): a test library, never the default
LIB_DEBUG_BOUNDS_PATH = os.path.join(BUILD_DIR, "libsgemm_debug_bounds.so")
HEADER = os.path.join(ROOT, "include", "sgemm.h")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMPILE_FLAGS = [
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
]
LINK_FLAGS = ["--shared", "-cudart", "static"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc")
    if not cand and os.path.exists("/usr/local/cuda/bin/nvcc"):
        cand = "/usr/local/cuda/bin/nvcc"
    if not cand:
        raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit on PATH")
    return cand


def units():
    """The library's translation units (compiled separately, in parallel)."""
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def sources():
    return sorted(units() + glob.glob(os.path.join(CSRC, "*.cuh")) + [HEADER])


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False, extra_flags=None,
          debug_bounds: bool = False) -> str:
    """Compile every translation unit to an object at the same time, then link
    libsgemm.so (no relocatable device code: each unit's kernels are complete).
    debug_bounds=True builds the range-checked test library instead
    (libsgemm_debug_bounds.so, -DSGEMM_DEBUG_BOUNDS)."""
    lib_path = LIB_DEBUG_BOUNDS_PATH if debug_bounds else LIB_PATH
    if not force and not is_stale(lib_path):
        return lib_path
    obj_dir = os.path.join(BUILD_DIR, f"obj{'_db' if debug_bounds else ''}{os.getpid()}")
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = [*ARCH_FLAGS, *COMPILE_FLAGS, *(extra_flags or []),
             *(["-DSGEMM_DEBUG_BOUNDS"] if debug_bounds else [])]
    if verbose:
        flags.insert(0, "-Xptxas=-v")

    def compile_unit(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.stdout or r.stderr:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise subprocess.CalledProcessError(r.returncode, cmd)
        return obj

    srcs = units()
    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_unit, srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *ARCH_FLAGS, *LINK_FLAGS, *objs, "-o", tmp], check=True)
    os.replace(tmp, lib_path)
    shutil.rmtree(obj_dir, ignore_errors=True)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
