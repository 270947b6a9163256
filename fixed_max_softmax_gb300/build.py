"""Build libfm.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel to an object file, then the
objects are linked into fixed_max_softmax_gb300/_build/libfm.so (static CUDA runtime).
Only the fm_* entry points of include/fm.h are exported.  build(debug=True) makes the same
library with -DFM_DEBUG in _build_debug/: the kernels' index checks on (FM_ERR_INDEX).
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libfm.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
SOURCES = ["fm_api.cu", "fm_bounds.cu", "fm_chunk_simt.cu", "fm_chunk_tc.cu", "fm_finalize.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                   "-I", os.path.join(ROOT, "include"), *extra]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    build_dir = BUILD_DEBUG if debug else BUILD
    lib = os.path.join(build_dir, "libfm.so")
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, "fm_internal.h"), os.path.join(ROOT, "include", "fm.h")]
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or ptxas_info or _stale(o, [s] + headers):
            extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DFM_DEBUG"] if debug else [])
            jobs.append([NVCC, *_flags(extra), "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stderr)
        return r

    with ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        run([NVCC, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv, debug="--debug" in sys.argv))
