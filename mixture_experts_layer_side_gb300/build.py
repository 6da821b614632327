"""Build libmok.so in-tree with nvcc for sm_103a (no CMake).

Each translation unit is compiled in parallel, then linked into
``mixture_experts_layer_side_gb300/libmok.so``.  Run ``python -m
mixture_experts_layer_side_gb300.build`` or call ``build()``.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libmok.so")
SOURCES = ["api.cu", "schedule.cu", "elementwise.cu", "gemm.cu", "mxfp8.cu", "router.cu", "ep.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmok.so")
    return path


def _compile(src, extra):
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *CFLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, res


def build(verbose=False, ptxas_info=False):
    """Compile every CUDA source and link libmok.so; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    objs = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        for src, obj, res in pool.map(lambda s: _compile(s, extra), SOURCES):
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
            if verbose or ptxas_info:
                sys.stderr.write(res.stderr)
            objs.append(obj)
    tmp = LIB_PATH + ".tmp"
    res = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
