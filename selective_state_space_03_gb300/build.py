"""Compile libssm_scan.so from csrc/*.cu for sm_103a (GB300) with nvcc.

Objects are rebuilt when a source or header is newer; translation units compile
in parallel. The library links the CUDA runtime statically, so it only needs the
driver at run time. Outputs, inside this package:

  _lib/libssm_scan.so          the library;
  _lib/libssm_scan_testing.so  the same kernels with the C ABI compiled with
                               SSM_SCAN_TESTING: schedule choices can then be
                               overridden through SSM_SCAN_FORCE_* variables,
                               for the tests that cover every schedule. The
                               release library has no such overrides.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libssm_scan.so")
TESTING_LIB = os.path.join(LIB_DIR, "libssm_scan_testing.so")
TESTING_SRC = "ssm_api.cu"          # the only translation unit that differs in the testing build

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libssm_scan.so")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(p) > t for p in deps)


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Build (if needed) both libraries and return the path of libssm_scan.so."""
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = _headers()
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(job):
        src, testing = job
        obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ("_testing.o" if testing else ".o"))
        if ptxas_info or _stale(obj, [src] + headers):
            defs = ["-DSSM_SCAN_TESTING"] if testing else []
            cmd = [cc] + NVCC_FLAGS + defs + extra + ["-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose or ptxas_info:
                print(r.stdout + r.stderr)
        return obj

    jobs = [(s, False) for s in srcs] + [(os.path.join(CSRC, TESTING_SRC), True)]
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, jobs))
    release = objs[:len(srcs)]
    testing = [o for s, o in zip(srcs, release) if os.path.basename(s) != TESTING_SRC] + [objs[-1]]
    for lib, parts in ((LIB, release), (TESTING_LIB, testing)):
        if _stale(lib, parts):
            tmp = lib + f".tmp{os.getpid()}"
            cmd = [cc] + ARCH + ["-shared", "-o", tmp] + parts
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
