"""Build the codec library ``libkvcodec.so`` in-tree with nvcc for sm_103a.

Translation units compile in parallel; the static CUDA runtime is linked in, so
the library loads (for symbol and host-only checks) on machines without a GPU.
``build(debug=True)`` builds ``libkvcodec_debug.so`` instead: the same sources
with -DKVC_BOUNDS_CHECK, whose kernels check every global access against the
call's buffers (a violation is skipped and the call returns KV_ERR_INTERNAL).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvcodec.so")
DEBUG_LIB = os.path.join(PKG, "libkvcodec_debug.so")
UNITS = ["fp8.cu", "uniform.cu", "turboquant.cu", "int8.cu", "crc.cu", "kv_codec_host.cpp"]
HEADERS = ["kv_internal.h", "device_common.cuh", "crc_common.cuh"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-ffp-contract=off", "-I", os.path.join(ROOT, "include"), "-I", SRC]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(unit, extra, out_dir):
    src = os.path.join(SRC, unit)
    obj = os.path.join(out_dir, unit + ".o")
    deps = [src, os.path.join(ROOT, "include", "kv_codec.h")] + [os.path.join(SRC, h) for h in HEADERS]
    if _stale(obj, deps + [__file__]):
        cmd = [NVCC] + ARCH + FLAGS + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {unit}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    out_dir = OUT_DIR + ("_debug" if debug else "")
    lib = DEBUG_LIB if debug else LIB
    os.makedirs(out_dir, exist_ok=True)
    if force:
        for f in os.listdir(out_dir):
            os.remove(os.path.join(out_dir, f))
    extra = (["-Xptxas", "-v"] if verbose_ptxas else []) + (["-DKVC_BOUNDS_CHECK"] if debug else [])
    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(lambda u: _compile(u, extra, out_dir), UNITS))
    if force or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list:
    """Both libraries, their translation units compiled side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        return list(ex.map(lambda d: build(force=force, debug=d), (False, True)))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
