"""Build the CUDA extension ``_lib/libmoe_gb300.so`` in-tree with nvcc.

One ``-gencode arch=compute_103a,code=sm_103a`` target (GB300), ``-O3
-lineinfo``, C++17; translation units compile in parallel and link into one
shared library with the CUDA runtime linked statically, so loading it needs
no library path setup. The library exports exactly the C ABI of
``include/moe.h``.

``build(debug_bounds=True)`` builds the bounds-checking variant
``_lib/libmoe_gb300_debug.so`` (``-DMOE_DEBUG_BOUNDS=1``: device-side checks
of the indices the kernels read from buffers, see ``moe_device_status``);
the binding loads it when the environment variable ``MOE_DEBUG_BOUNDS`` is 1.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libmoe_gb300.so")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_DEBUG = os.path.join(OUT_DIR, "libmoe_gb300_debug.so")
OBJ_DIR_DEBUG = os.path.join(PKG, "_build_debug")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
         "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(CSRC, "*.h")) +
            [os.path.join(ROOT, "include", "moe.h"), os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, jobs: int | None = None,
          debug_bounds: bool = False) -> str:
    """Compile (if needed) and return the path of the shared library (the
    bounds-checking variant with debug_bounds)."""
    lib = LIB_DEBUG if debug_bounds else LIB
    obj_dir = OBJ_DIR_DEBUG if debug_bounds else OBJ_DIR
    extra = ["-DMOE_DEBUG_BOUNDS=1"] if debug_bounds else []
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(obj_dir, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
