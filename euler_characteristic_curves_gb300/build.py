"""Builds the CUDA library libecc_gb300.so in-tree (euler_characteristic_curves_gb300/_build/).

Every translation unit is compiled by nvcc for sm_103a only, in parallel, then linked into one
shared library with the CUDA runtime linked statically, so loading the library needs no other
CUDA shared object than the driver.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libecc_gb300.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
# The debug variant: the same sources with ECC_DEBUG_BOUNDS=1 (bounds checks that record a bit
# in the device error word and skip the access), loaded by the binding when ECC_DEBUG=1.
DEBUG_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_DIR, "libecc_gb300_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-ffp-contract=off", "--expt-relaxed-constexpr"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the ECC library needs the CUDA toolkit to build")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    deps = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    deps.append(os.path.join(INCLUDE, "ecc.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile and link the library (``debug``: the bounds-checked variant); returns its path.
    Skips work when nothing changed."""
    build_dir, lib_path = (DEBUG_DIR, DEBUG_LIB_PATH) if debug else (BUILD_DIR, LIB_PATH)
    if debug:
        extra_flags = (*extra_flags, "-DECC_DEBUG_BOUNDS=1")
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-I", CSRC, "-c", src,
               "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(sources()))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else [],
                debug="--debug" in sys.argv))
