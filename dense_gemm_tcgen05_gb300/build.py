"""In-tree build of libgemm.so (nvcc, sm_103a only).

Each translation unit is compiled in parallel to an object file under
``_build/``; the objects are linked into ``libgemm.so`` beside this file with
the CUDA runtime linked statically, so the library needs only the NVIDIA
driver at run time.  ``python -m dense_gemm_tcgen05_gb300.build [-v]``
rebuilds when a source is newer than the library; ``-v`` adds ``-Xptxas -v``
(registers, shared memory, spills) to the log in ``_build/``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgemm.so")

SOURCES = ["api.cu", "tc_gemm_f16.cu", "tc_gemm_bf16.cu", "tc_gemm_bf16f32.cu", "tc_gemm_fp8.cu",
           "simt_f32.cu", "split_f32.cu", "misc_kernels.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libgemm.so")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "gemm.h"))
    files.append(os.path.abspath(__file__))
    return files


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src: str, ptxas_verbose: bool) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".log")
    with open(log, "w") as fh:
        fh.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s" % (src, res.stderr[-6000:]))
    return obj


def build(force: bool = False, ptxas_verbose: bool = False, jobs: int | None = None) -> str:
    """Compile libgemm.so if it is missing or stale; returns its path."""
    if not force and not ptxas_verbose and not is_stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    jobs = jobs or min(len(SOURCES), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, ptxas_verbose), SOURCES))
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s" % res.stderr[-6000:])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    verbose = "-v" in sys.argv
    path = build(force=True, ptxas_verbose=verbose)
    print(path)
    if verbose:
        for src in SOURCES:
            log = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".log")
            print(open(log).read())
