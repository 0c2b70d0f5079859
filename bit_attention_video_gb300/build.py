"""In-tree build of ``libvca.so`` (the C ABI of ``include/vca.h``) for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library with the CUDA runtime linked statically.  No torch extension
machinery is involved: the library has a plain C ABI.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libvca.so")
# The debug build: the same sources with -DVCA_DEBUG, whose kernels check the
# data-dependent indices they address memory with (a cached permutation, a
# label) and record an error instead of reading or writing out of bounds.
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libvca.so")
SOURCES = ["api.cu", "prep.cu", "attn_fp8.cu", "attn_bf16.cu", "attn_nvfp4.cu", "debug.cu",
           "pipeline.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-diag-suppress", "177"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libvca.so")


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hdrs + [os.path.join(ROOT, "include", "vca.h")]


def _stale(target, inputs) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(i) > t for i in inputs)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile libvca.so (debug=True: the -DVCA_DEBUG build in its own folder)."""
    out_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    deps = _deps()
    objs, jobs = [], []
    flags = FLAGS + (["-DVCA_DEBUG"] if debug else [])
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + deps):
            jobs.append([nvcc, *ARCH, *flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return cmd[-3], r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for src, log in ex.map(run, jobs):
            with open(os.path.join(out_dir, os.path.basename(src) + ".ptxas.txt"), "w") as f:
                f.write(log)
            if verbose:
                print(log)
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))
