"""Build ``libccl.so`` (CUDA executor + host compiler) for sm_103a with nvcc.

Translation units are compiled in parallel and linked into a shared library
next to this file; nothing is installed.  Rebuilds only what changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libccl.so")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["ccl_runtime.cu", "ccl_static.cu", "ccl_compiler.cpp", "ccl_builtin.cpp", "ccl_planner.cpp",
           "ccl_tuner.cpp", "ccl_persist.cpp"]
HEADERS = ["ccl_internal.h", "ccl_plan.h", "ccl_executor.cuh", "ccl_device.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nvcc: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib", "lib"):
        d = os.path.join(root, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return os.path.join(root, "lib64")


def _newest_dep_mtime() -> float:
    files = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "ccl.h")]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    dep_t = _newest_dep_mtime()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src + ".o")
        objs.append(o)
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), dep_t):
            jobs.append([nvcc, *ARCH, *COMMON, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return cmd[-1]

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(run, jobs))
    if jobs or force or not os.path.exists(LIB) or \
            os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        libdir = _cuda_lib_dir(nvcc)
        tmp = LIB + ".tmp"
        run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
             "-Xlinker", "-rpath", "-Xlinker", libdir])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
