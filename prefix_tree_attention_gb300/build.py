"""Build ``libtreeattn.so`` in-tree for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a``; the host packer is plain
C++.  The shared library lands next to this file in ``lib/`` and is what the
Python binding loads.  Run ``python prefix_tree_attention_gb300/build.py`` (by path:
importing the package needs the library this script produces).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "lib")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libtreeattn.so"
DEBUG_LIB_NAME = "libtreeattn_debug.so"     # the same sources with TREE_DEBUG
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

CUDA_SOURCES = ["api.cu", "positions.cu", "blockmap.cu", "attn_fwd.cu", "attn_bwd.cu",
                "diag.cu", "logprob.cu", "dta_attn.cu", "lmhead.cu"]
CXX_SOURCES = ["packer.cpp", "partition.cpp", "dta.cpp"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    """Compile every source and link the shared library; returns its path.
    ``debug`` builds the bounds-checked variant (``-DTREE_DEBUG``) as
    ``libtreeattn_debug.so`` next to the release library."""
    build_dir = BUILD_DIR + ("_debug" if debug else "")
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    cuda_flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                         "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr"]
    if debug:
        cuda_flags += ["-DTREE_DEBUG"]
    if ptxas_info:
        cuda_flags += ["-Xptxas", "-v"]
    jobs = []
    objs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(build_dir, src + ".o")
        objs.append(obj)
        jobs.append([nvcc] + cuda_flags + ["-c", os.path.join(CSRC, src), "-o", obj])
    for src in CXX_SOURCES:
        obj = os.path.join(build_dir, src + ".o")
        objs.append(obj)
        jobs.append([nvcc, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler",
                     "-fvisibility=hidden", "-c", os.path.join(CSRC, src), "-o", obj])
    with ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        logs = list(ex.map(_run, jobs))
    if verbose or ptxas_info:
        for log in logs:
            if log.strip():
                print(log)
    out = os.path.join(OUT_DIR, DEBUG_LIB_NAME if debug else LIB_NAME)
    tmp = out + ".tmp"
    _run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    path = build(verbose=True, ptxas_info="--ptxas" in sys.argv, debug="--debug" in sys.argv)
    print(path)
