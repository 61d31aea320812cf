"""Build libtreeattn.so in-tree for sm_103a (nvcc + g++, no cmake).

    python -m tree_structured_decode_gb300.build

Translation units compile in parallel; the shared library links the CUDA
runtime statically, so it needs only the CUDA driver library (libcuda) at
run time.  Output:
``tree_structured_decode_gb300/lib/libtreeattn.so``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libtreeattn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _nvcc():
    p = os.path.join(CUDA_HOME, "bin", "nvcc")
    return p if os.path.exists(p) else (shutil.which("nvcc") or "nvcc")


def _units(extra_nvcc):
    inc = ["-I", os.path.join(os.path.dirname(PKG), "include"), "-I", CSRC]
    cu = [_nvcc(), "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
          "--expt-relaxed-constexpr", *inc, *extra_nvcc]
    cxx = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-Wno-unused-function",
           "-I", os.path.join(CUDA_HOME, "include"), *inc]
    jobs = []
    for name in sorted(os.listdir(CSRC)):
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD, name + ".o")
        if name.endswith(".cu"):
            jobs.append((cu + ["-c", src, "-o", obj], obj))
        elif name.endswith(".cpp"):
            jobs.append((cxx + ["-c", src, "-o", obj], obj))
    return jobs


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    return cmd, r


def build(verbose: bool = False, extra_nvcc=()) -> str:
    """Compile every translation unit and link the library; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    jobs = _units(list(extra_nvcc))
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(lambda j: _run(j[0]), jobs))
    for cmd, r in results:
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {cmd[-3]}")
    tmp = LIB + ".tmp"
    link = [_nvcc(), "-shared", *ARCH, "-o", tmp] + [o for _, o in jobs] + ["-lpthread", "-ldl", "-lrt"]
    cmd, r = _run(link)
    if verbose or r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
