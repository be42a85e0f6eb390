"""Builds the native library in-tree: prefix_shared_kv_gb300/_lib/librx.so.

Every CUDA source is compiled for sm_103a only (``-gencode arch=compute_103a,code=sm_103a``;
the ``a`` target is needed for tcgen05 / TMA), host sources with g++; translation units are
compiled in parallel and linked with nvcc.  Run ``python -m prefix_shared_kv_gb300.build``.
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
OUT = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT, "librx.so")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc") if os.path.exists(
    os.path.join(CUDA_HOME, "bin", "nvcc")) else (shutil.which("nvcc") or "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC, "--expt-relaxed-constexpr"]
CXX_FLAGS = ["-O2", "-fPIC", "-std=c++17", "-Wall", "-I" + INCLUDE, "-I" + CSRC,
             "-I" + os.path.join(CUDA_HOME, "include")]


def _sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(f for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(verbose: bool = False, extra_nvcc=()) -> str:
    cu, cpp = _sources()
    obj_dir = os.path.join(OUT, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    jobs = []
    for f in cu:
        o = os.path.join(obj_dir, f + ".o")
        jobs.append([NVCC, *NVCC_FLAGS, *extra_nvcc, "-c", os.path.join(CSRC, f), "-o", o])
    for f in cpp:
        o = os.path.join(obj_dir, f + ".o")
        jobs.append([shutil.which("g++") or "g++", *CXX_FLAGS, "-c", os.path.join(CSRC, f),
                     "-o", o])
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(_run, jobs))
    if verbose:
        for log in logs:
            if log.strip():
                print(log)
    objs = [j[-1] for j in jobs]
    tmp = LIB + ".tmp"
    _run([NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
          "-Xlinker", "-rpath," + os.path.join(CUDA_HOME, "lib64")])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
