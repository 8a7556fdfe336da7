"""Build libtq.so in-tree: nvcc for the sm_103a kernels, g++ for the host core.

Usage: ``python -m turboquant_paged_kv_gb300.build`` (or ``build()``). The
library lands in ``turboquant_paged_kv_gb300/_lib/libtq.so``; objects go to
``_build/`` at the repository root. Both are git-ignored build products.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(ROOT, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libtq.so")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]

CU_SOURCES = ["tq_store.cu", "tq_decode.cu", "tq_decode_noalloc.cu", "tq_dequant.cu", "tq_prod.cu",
              "tq_prod_store.cu", "tq_continue.cu"]
CPP_SOURCES = ["tq_host.cpp"]


def _sources():
    return [os.path.join(CSRC, s) for s in CU_SOURCES + CPP_SOURCES]


def _deps():
    return _sources() + [os.path.join(CSRC, "tq_internal.h"), os.path.join(CSRC, "tq_launch.cuh"),
                         os.path.join(CSRC, "tq_vec.cuh"), os.path.join(CSRC, "tq_attn.cuh"),
                         os.path.join(CSRC, "tq_prod.cuh"), os.path.join(CSRC, "tq_store.cuh"),
                         os.path.join(INCLUDE, "tq.h"),
                         os.path.abspath(__file__)]


def _up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _run(cmd):
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if proc.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + proc.stdout)
    return proc.stdout


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libtq.so; returns its path."""
    if not force and _up_to_date():
        return LIB_PATH
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    jobs = []
    for s in CU_SOURCES:
        obj = os.path.join(OBJ_DIR, s + ".o")
        jobs.append((obj, [NVCC] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else [])
                     + ["-c", os.path.join(CSRC, s), "-o", obj]))
    cxx = shutil.which("g++") or "c++"
    for s in CPP_SOURCES:
        obj = os.path.join(OBJ_DIR, s + ".o")
        jobs.append((obj, [cxx] + CXX_FLAGS + ["-c", os.path.join(CSRC, s), "-o", obj]))
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(lambda j: _run(j[1]), jobs))
    if verbose:
        for o in outs:
            sys.stdout.write(o)
    tmp = LIB_PATH + ".tmp"
    _run([NVCC] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + [j[0] for j in jobs]
         + ["-Xlinker", "-rpath," + os.path.join(CUDA_HOME, "lib64")])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
