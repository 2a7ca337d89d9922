"""Build the sm_103a shared library ``_build/libulysses_gb300.so`` in-tree.

Each ``csrc/*.cu`` is compiled by nvcc in parallel (one ``-gencode`` for
sm_103a, ``-lineinfo``), then linked with ``nvcc -shared``.  The CUDA runtime
is linked statically; the driver's tensor-map encoder is resolved at run time,
so the library needs no ``-lcuda``.  Run as ``python -m
long_context_sequence_head_gb300.build`` or through ``__graft_entry__.build()``.

``build(debug=True)`` compiles the same sources with ``-DULY_DEBUG`` into
``_build/debug/libulysses_gb300_debug.so``: every raw-pointer global access of
the swap and attention kernels is checked against its buffer and a failure is
reported as a status (ULY_ERR_BOUNDS) instead of being made.  The binding
loads it when ULY_DEBUG_BUILD=1.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
SO_NAME = "libulysses_gb300.so"
SO_PATH = os.path.join(BUILD, SO_NAME)
DEBUG_BUILD = os.path.join(BUILD, "debug")
DEBUG_SO_PATH = os.path.join(DEBUG_BUILD, "libulysses_gb300_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))) + [
        os.path.join(ROOT, "include", "ulysses.h")]


def up_to_date(debug: bool = False) -> bool:
    so = DEBUG_SO_PATH if debug else SO_PATH
    if not os.path.exists(so):
        return False
    t = os.path.getmtime(so)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    so_path = DEBUG_SO_PATH if debug else SO_PATH
    out_dir = DEBUG_BUILD if debug else BUILD
    if not force and up_to_date(debug):
        return so_path
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-I", os.path.join(ROOT, "include"), "-I", CSRC] + (["-DULY_DEBUG"] if debug else [])
    objs = []

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + common + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = so_path + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, so_path)
    return so_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
