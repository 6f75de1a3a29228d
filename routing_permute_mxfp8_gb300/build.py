"""Builds libmm_moe.so (CUDA, sm_103a) in-tree, and its checked build
libmm_moe_check.so (the same sources with MM_CHECK: device index checks).

Each translation unit under csrc/ is compiled in parallel with nvcc for
sm_103a only (both variants at once), then linked into a shared library
against the shared CUDA runtime.  Usage: ``python -m routing_permute_mxfp8_gb300.build``.
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
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmm_moe.so")
OBJ_CHECK = os.path.join(PKG, "_build_check")
LIB_CHECK = os.path.join(PKG, "libmm_moe_check.so")
SOURCES = ["route.cu", "permute.cu", "gemm.cu", "combine.cu", "abi.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libmm_moe.so")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


# (library, object directory, extra flags): the library and its checked
# build (MM_CHECK: device index checks that report MM_DEVERR_BOUNDS)
VARIANTS = [(LIB, OBJ, []), (LIB_CHECK, OBJ_CHECK, ["-DMM_CHECK=1"])]


def build(verbose: bool = False, extra_flags=()) -> str:
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                    "--expt-relaxed-constexpr"] + list(extra_flags)

    def compile_one(job):
        src, obj_dir, vflags = job
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + flags + vflags
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    jobs = []
    for _, obj_dir, vflags in VARIANTS:
        os.makedirs(obj_dir, exist_ok=True)
        jobs += [(src, obj_dir, vflags) for src in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    libdir = _cuda_lib_dir(nvcc)
    for i, (lib, _, _) in enumerate(VARIANTS):
        tmp = lib + ".tmp"
        cmd = [nvcc, "-shared", "-o", tmp] + objs[i * len(SOURCES):(i + 1) * len(SOURCES)] + ARCH + \
            ["-cudart", "shared", "-Xlinker", f"-rpath,{libdir}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
