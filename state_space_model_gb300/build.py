"""Builds ``libssd_gb300.so`` in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel into
``_build/``; the shared library links the CUDA runtime statically so it
loads on a machine without a GPU driver (nothing touches the driver until
the first CUDA call).  Usage: ``python -m state_space_model_gb300.build``.

``--debug-bounds`` builds ``libssd_gb300_debug.so`` instead (objects in
``_build_debug/``), compiled with ``-DSSD_DEBUG_BOUNDS``: the kernels check
every index, shared-memory offset and tensor-memory column range they compute
and report failures through ssd_device_status (see csrc/ssd_debug.cuh).
Python loads it when SSD_DEBUG_BOUNDS=1 is set.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libssd_gb300.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libssd_gb300_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libssd_gb300")
    return exe


def _flags(verbose_ptxas: bool, debug_bounds: bool = False) -> list[str]:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                "--expt-relaxed-constexpr"]
    if debug_bounds:
        f += ["-DSSD_DEBUG_BOUNDS"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) +
                  glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps() -> list[str]:
    return (_sources() + glob.glob(os.path.join(CSRC, "*.h")) +
            glob.glob(os.path.join(CSRC, "*.cuh")) +
            [os.path.join(ROOT, "include", "ssd.h"), os.path.abspath(__file__)])


def up_to_date(debug_bounds: bool = False) -> bool:
    lib = LIB_DEBUG if debug_bounds else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose_ptxas: bool | None = None,
          debug_bounds: bool = False) -> str:
    lib = LIB_DEBUG if debug_bounds else LIB
    out_dir = BUILD_DEBUG if debug_bounds else BUILD
    if not force and up_to_date(debug_bounds):
        return lib
    if verbose_ptxas is None:
        verbose_ptxas = os.environ.get("SSD_PTXAS_VERBOSE", "0") == "1"
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = _flags(verbose_ptxas, debug_bounds)

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose_ptxas and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
