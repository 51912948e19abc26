"""Builds the in-tree C-ABI library ``_lib/libhstu_attn.so`` for sm_103a.

Each CUDA translation unit is compiled by nvcc in parallel, then linked into
one shared library (CUDA runtime linked statically; the tensor-map encoder is
fetched from the driver at run time).  Rebuilds only when a source or header
is newer than the library.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libhstu_attn.so")

SOURCES = ["hstu_api.cu", "hstu_sched.cu", "hstu_fwd_d64.cu", "hstu_fwd_d96.cu", "hstu_fwd_d128.cu", "hstu_fwd_pair_d128.cu", "hstu_fwd_d256.cu",
           "hstu_static_ws.cu", "hstu_bwd_d64.cu", "hstu_bwd_d96.cu", "hstu_bwd_d128.cu",
           "hstu_fwd_rab_d64.cu", "hstu_fwd_rab_d96.cu", "hstu_fwd_rab_d128.cu", "hstu_fwd_rab_d256.cu",
           "hstu_bwd_rab_d64.cu", "hstu_bwd_rab_d96.cu", "hstu_bwd_rab_d128.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library; returns its path."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        out = _run([nvcc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj])
        return obj, out

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, out in results:
            sys.stdout.write(out)
    tmp = LIB_PATH + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
