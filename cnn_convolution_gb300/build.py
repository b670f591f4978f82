"""Build libconv2d_gb300.so in-tree with nvcc for sm_103a.

Every translation unit is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically; the driver API entry points
needed for tensor maps are resolved at run time, so the library has no link
dependency on libcuda.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
# One build folder per host architecture, so objects from another machine are never linked.
BUILD_DIR = os.path.join(PKG, "_build", platform.machine())
LIB_NAME = "libconv2d_gb300.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)

SOURCES = ["api.cpp", "status.cu", "cuda_core_conv.cu", "tc_conv_sm103a.cu", "tf32x3_conv_sm103a.cu",
           "direct_conv.cu", "signature.cu", "deconv.cu", "peaks.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA library cannot be built")
    return cand


def _flags(src: str):
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if src.endswith(".cu"):
        return common + ARCH + ["-lineinfo", "--expt-relaxed-constexpr", "-Xptxas", "-v"]
    return common


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = nvcc_path()
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "conv2d.h"))
    objs, jobs = [], []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        op = os.path.join(BUILD_DIR, src + ".o")
        objs.append(op)
        if force or not _newer(op, [sp] + headers):
            jobs.append((sp, op))

    def compile_one(job):
        sp, op = job
        cmd = [nvcc, "-c", sp, "-o", op] + _flags(sp)
        r = subprocess.run(cmd, capture_output=True, text=True)
        return sp, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for sp, r in ex.map(compile_one, jobs):
                if verbose or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {os.path.basename(sp)}")
                log = os.path.join(BUILD_DIR, os.path.basename(sp) + ".ptxas.txt")
                with open(log, "w") as f:
                    f.write(r.stdout + r.stderr)
    if force or jobs or not _newer(LIB_PATH, objs):
        tmp = LIB_PATH + f".{os.getpid()}.tmp"
        cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
