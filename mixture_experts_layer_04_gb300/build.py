"""Build the CUDA library libmoe_gb300.so in-tree for sm_103a.

Each translation unit under csrc/ is compiled by nvcc in parallel
(-gencode arch=compute_103a,code=sm_103a) and linked into one shared library with
the CUDA runtime linked statically.  Objects and the library go to ``_build/`` next
to this file.  A unit is rebuilt when it or any header under csrc/ or include/ is
newer than its object.

``build(debug=True)`` compiles the same sources with -DMOE_DEBUG into ``_build_debug/``:
that library's kernels check the indices they take from their inputs (expert ids, group
offsets, row maps) and report a bad one through moe_sync_check() instead of using it.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_NAME = "libmoe_gb300.so"
LIB_PATH = os.path.join(BUILD, LIB_NAME)
LIB_PATH_DEBUG = os.path.join(BUILD_DEBUG, LIB_NAME)

SOURCES = ["api.cu", "route.cu", "permute.cu", "combine.cu", "gemm_tc.cu",
           "permute_noalloc.cu", "route_cluster.cu", "capacity.cu", "quant.cu",
           "gemm_tf32.cu"]
GENCODE = "-gencode=arch=compute_103a,code=sm_103a"
NVCC_FLAGS = [
    GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
    "--expt-relaxed-constexpr", "-Xptxas", "-v" if os.environ.get("MOE_PTXAS_VERBOSE") else "-O3",
]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libmoe_gb300")
    return cand


def _headers_mtime() -> float:
    m = 0.0
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".h", ".cuh")):
                m = max(m, os.path.getmtime(os.path.join(d, f)))
    return m


def _compile(src: str, hdr_mtime: float, force: bool, out_dir: str, extra: list) -> str:
    s = os.path.join(CSRC, src)
    o = os.path.join(out_dir, src.replace(".cu", ".o"))
    if (not force and os.path.exists(o) and os.path.getmtime(o) >= os.path.getmtime(s)
            and os.path.getmtime(o) >= hdr_mtime):
        return o
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-I", INCLUDE, "-c", s, "-o", o]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if os.environ.get("MOE_PTXAS_VERBOSE"):
        sys.stderr.write(r.stderr)
    return o


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile every CUDA unit and link libmoe_gb300.so; returns the library path.
    With ``debug`` the library is the bounds-checking build under _build_debug/."""
    out_dir = BUILD_DEBUG if debug else BUILD
    lib_path = LIB_PATH_DEBUG if debug else LIB_PATH
    extra = ["-DMOE_DEBUG"] if debug else []
    os.makedirs(out_dir, exist_ok=True)
    hm = _headers_mtime()
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, hm, force, out_dir, extra), SOURCES))
    newest = max(os.path.getmtime(o) for o in objs)
    if force or not os.path.exists(lib_path) or os.path.getmtime(lib_path) < newest:
        tmp = lib_path + ".tmp"
        cmd = [nvcc(), GENCODE, "-shared", "-o", tmp, *objs, "-cudart", "static", "-ldl"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    if verbose:
        print(lib_path)
    return lib_path


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv)
