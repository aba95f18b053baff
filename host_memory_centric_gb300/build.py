"""Builds libmt.so in-tree for sm_103a (nvcc for the kernels, g++ for host code).

Run as ``python -m host_memory_centric_gb300.build``.  Translation units are
compiled in parallel; the result is ``host_memory_centric_gb300/libmt.so``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libmt.so")
BUILD = os.path.join(ROOT, "_build")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA, "bin", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

CU_SRCS = ["k_gemm.cu", "k_attention.cu", "k_attention_tc.cu", "k_elementwise.cu", "k_noalloc.cu", "k_moe.cu"]
CPP_SRCS = ["mt_runtime.cpp", "mt_host.cpp"]
HEADERS = ["mt_kernels.h", "mt_host.h"]


def _newest_input() -> float:
    files = [os.path.join(SRC, f) for f in CU_SRCS + CPP_SRCS + HEADERS]
    files.append(os.path.join(ROOT, "include", "mt.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(OUT) and os.path.getmtime(OUT) >= _newest_input():
        return OUT
    os.makedirs(BUILD, exist_ok=True)
    inc = ["-I" + os.path.join(ROOT, "include"), "-I" + SRC]
    jobs = []
    for f in CU_SRCS:
        o = os.path.join(BUILD, f + ".o")
        jobs.append((o, [NVCC, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                         "-Xptxas", "-v" if verbose else "-O3", *inc, "-c", os.path.join(SRC, f), "-o", o]))
    cxx = shutil.which("g++") or "g++"
    for f in CPP_SRCS:
        o = os.path.join(BUILD, f + ".o")
        jobs.append((o, [cxx, "-O3", "-std=c++17", "-fPIC", "-fno-math-errno", "-Wall",
                         "-I" + os.path.join(CUDA, "include"), *inc, "-c", os.path.join(SRC, f), "-o", o]))
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        logs = list(ex.map(lambda j: _run(j[1]), jobs))
    if verbose:
        for l in logs:
            sys.stdout.write(l)
    tmp = OUT + ".tmp"
    _run([NVCC, *ARCH, "-shared", "-o", tmp, *[j[0] for j in jobs], "-lpthread"])
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
