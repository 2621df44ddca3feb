"""Build libmoe_gb300.so in-tree with nvcc for sm_103a (GB300).

A host generator (``csrc/silu_table_gen.cpp``, built with the system C++
compiler) first writes the activation kernel's SiLU table into the build
folder; then each ``csrc/*.cu`` compiles to an object file in parallel, and
nvcc links the shared library next to this file.  The CUDA runtime is linked
statically, so the library needs only the driver at run time.

    python -m combine_moe_dispatch_gb300.buildlib [--verbose-ptxas] [--force]
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=default",
                 "-I", INCLUDE, "-I", CSRC, "-I", BUILD_DIR]
TABLE_GEN = os.path.join(CSRC, "silu_table_gen.cpp")
TABLE = os.path.join(BUILD_DIR, "silu_table.inc")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h"))) + [TABLE_GEN]


def generate_table(cxx: str = "g++") -> str:
    """Compile and run the SiLU table generator (plain IEEE binary32: no
    fused contraction, no fast-math)."""
    exe = os.path.join(BUILD_DIR, "silu_table_gen")
    cmd = [cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-o", exe, TABLE_GEN]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"{cxx} failed on {TABLE_GEN}:\n{r.stdout}\n{r.stderr}")
    r = subprocess.run([exe, TABLE], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"silu_table_gen failed:\n{r.stdout}\n{r.stderr}")
    return TABLE


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs() + [__file__])


def build(force: bool = False, verbose_ptxas: bool = False, nvcc: str = "nvcc") -> str:
    if not force and not verbose_ptxas and up_to_date():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    generate_table()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        cmd = [nvcc, *CFLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose_ptxas:
            sys.stderr.write(r.stderr)
        return obj

    srcs = _sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--verbose-ptxas" in sys.argv))
