"""Build step for the CUDA libraries (nvcc, sm_103a only).

Compiles ``csrc/*.cu`` in parallel into ``_build/`` and links
``libmc2_gb300.so`` (the operations) next to this file, and ``calib/*.cu``
into ``libmc2_calib.so`` (a measurement probe that only the benchmark loads).
Rebuilds a library only when one of its sources or the public header is newer
than it.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
CALIB = os.path.join(HERE, "calib")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmc2_gb300.so")
CALIB_LIB = os.path.join(HERE, "libmc2_calib.so")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def sources(src_dir=CSRC):
    return sorted(glob.glob(os.path.join(src_dir, "*.cu")))


def _deps(src_dir=CSRC):
    return sources(src_dir) + glob.glob(os.path.join(src_dir, "*.cuh")) + glob.glob(os.path.join(src_dir, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)]


def needs_build(lib=LIB, src_dir=CSRC) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in _deps(src_dir))


def _build_one(lib, src_dir, force, verbose, extra_flags):
    if not force and not needs_build(lib, src_dir):
        return lib
    os.makedirs(BUILD, exist_ok=True)
    nvcc = NVCC if os.path.exists(NVCC) else "nvcc"
    srcs = sources(src_dir)
    tag = os.path.basename(src_dir)

    def compile_one(src):
        obj = os.path.join(BUILD, f"{tag}_{os.path.basename(src)}.o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Build the operations library (and return its path)."""
    return _build_one(LIB, CSRC, force, verbose, extra_flags)


def build_calib(force: bool = False, verbose: bool = False) -> str:
    """Build the benchmark's calibration probe library (and return its path)."""
    return _build_one(CALIB_LIB, CALIB, force, verbose, ())


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
    print(build_calib(force="--force" in sys.argv, verbose=True))
