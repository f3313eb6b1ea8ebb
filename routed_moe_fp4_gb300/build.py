"""Builds libcolimoe.so (the C-ABI library) from csrc/ with nvcc for sm_103a.

Translation units compile in parallel; the shared library lands in routed_moe_fp4_gb300/_lib/.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIB_DIR, "libcolimoe.so")
# The bounds-checked debug build (-DCOLI_BOUNDS_CHECK): the FP4 GEMM checks every tile record
# against the buffers, records kErrBounds and skips the tile instead of reading or writing outside.
LIB_CHECKED = os.path.join(LIB_DIR, "libcolimoe_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libcolimoe.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "colimoe.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, bounds_check: bool = False) -> str:
    """Builds libcolimoe.so, or with bounds_check the debug library libcolimoe_checked.so (the same
    sources with -DCOLI_BOUNDS_CHECK, objects in their own folder). Returns the library's path."""
    lib = LIB_CHECKED if bounds_check else LIB
    if not force and not _stale(lib):
        return lib
    os.makedirs(LIB_DIR, exist_ok=True)
    obj_dir = os.path.join(LIB_DIR, "obj_checked" if bounds_check else "obj")
    os.makedirs(obj_dir, exist_ok=True)
    nv = nvcc()
    extra = ["-DCOLI_BOUNDS_CHECK"] if bounds_check else []

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nv, *ARCH, *FLAGS, *extra, "-Xptxas", "-v" if verbose else "-O3", "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nv, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart", "-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, bounds_check="--bounds-check" in sys.argv))
