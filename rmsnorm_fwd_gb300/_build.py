"""Builds librmsnorm.so (the CUDA kernels + C ABI) in-tree with nvcc.

One nvcc process per translation unit, run in parallel, then one link.
Kernels are compiled for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``).  Output:
``rmsnorm_fwd_gb300/_build/librmsnorm.so`` (git-ignored).
"""
from __future__ import annotations

import fcntl
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "librmsnorm.so")

SOURCES = ["api.cpp", "select.cpp", "generic.cu", "staged.cu", "qknorm.cu", "cluster.cu",
           "gridrow.cu",
           "rowreg_f32.cu", "rowreg_bf16.cu", "rowreg_f16.cu",
           "rowreg_epi_f32.cu", "rowreg_epi_bf16.cu", "rowreg_epi_f16.cu",
           "rowreg_fp4_f32.cu", "rowreg_fp4_bf16.cu", "rowreg_fp4_f16.cu"]
HEADERS = ["internal.h", "host_link.h", "device_common.cuh", "rowreg.cuh"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC"]
CUDA_FLAGS = ["-lineinfo"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librmsnorm.so")


def _cuda_home(nvcc: str) -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    paths += [os.path.join(INCLUDE, "rmsnorm.h"), __file__]
    return max(os.path.getmtime(p) for p in paths)


def _fresh() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of librmsnorm.so.  Processes
    that build at the same time (parallel test workers) take turns on a lock
    file, so no two write the same object files; a process that waited finds
    the library fresh and returns it."""
    if not force and _fresh():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    with open(os.path.join(OUT, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and _fresh():
                return LIB
            return _build_locked(verbose)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(verbose: bool) -> str:
    nvcc = _nvcc()
    common = [*CFLAGS, "-I", INCLUDE, "-I", CSRC]

    def compile_one(src: str) -> str:
        obj = os.path.join(OUT, src + ".o")
        cmd = [nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cu"):
            cmd[1:1] = [*GENCODE, *CUDA_FLAGS]
            if verbose:
                cmd.append("-Xptxas=-v")
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    cuda_lib = os.path.join(_cuda_home(nvcc), "lib64")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", *GENCODE, "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath,{cuda_lib}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
