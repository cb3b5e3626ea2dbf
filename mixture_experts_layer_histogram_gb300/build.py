"""Builds libmoe.so (the CUDA kernels + C ABI) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel into ``_build/`` and linked as a shared library
next to this file. Up-to-date objects are reused.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmoe.so")
LIB_CHECKS = os.path.join(PKG, "libmoe_checks.so")
SOURCES = ["route_index.cu", "permute_combine.cu", "gemm_simt.cu", "gemm_tc.cu", "gemm_rows.cu", "router.cu", "api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nvcc):
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs.append(os.path.join(INCLUDE, "moe.h"))
    return max(os.path.getmtime(h) for h in hdrs)


def build(force: bool = False, verbose: bool = False, extra_flags=(), checks: bool = False) -> str:
    """checks=True: the debug build with the device-side consistency checks (-DMOE_CHECKS=1), written to
    libmoe_checks.so next to the release library."""
    nvcc = _nvcc()
    out_dir = os.path.join(BUILD, "checks") if checks else BUILD
    lib_path = LIB_CHECKS if checks else LIB
    os.makedirs(out_dir, exist_ok=True)
    dep_t = _deps()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}", f"-I{CSRC}",
                    "--expt-relaxed-constexpr"] + (["-DMOE_CHECKS=1"] if checks else []) + list(extra_flags) + \
        os.environ.get("MOE_NVCC_FLAGS", "").split()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), dep_t):
            jobs.append([nvcc] + flags + ["-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for out in ex.map(run, jobs):
            if verbose and out.strip():
                print(out)
    newest = max(os.path.getmtime(o) for o in objs)
    if force or jobs or not os.path.exists(lib_path) or os.path.getmtime(lib_path) < newest:
        libdir = _cuda_lib_dir(nvcc)
        tmp = lib_path + f".tmp{os.getpid()}"
        run([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs +
            ["-Xlinker", f"-rpath={libdir}", f"-L{libdir}"])
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
