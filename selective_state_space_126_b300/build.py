"""Builds libssm.so (the C-ABI library) in-tree with nvcc for sm_103a.

Usage: ``python -m selective_state_space_126_b300.build [--force]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libssm.so")
SOURCES = ["ssm_api.cu", "scan_generic.cu", "scan_tiled.cu", "scan_warp.cu", "state_update.cu", "conv1d.cu", "scan_bwd.cu",
           "probe.cu", "ssd.cu"]
HEADERS = ["device_math.cuh", "async_copy.cuh", "scan_common.cuh", "ssm_internal.h", "tcgen05.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                     "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "ssm.h"))
    files.append(os.path.abspath(__file__))
    return files


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build_library(force: bool = False, quiet: bool = False, extra_flags=(), verbose_ptxas: bool = False,
                  out: str = LIB) -> str:
    """Compile every CUDA source and link libssm.so; returns its path."""
    if not force and not is_stale(out):
        return out
    flags = list(NVCC_FLAGS) + list(extra_flags)
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    tmp = tempfile.mkdtemp(prefix="ssm_build_")
    try:
        def compile_one(src):
            obj = os.path.join(tmp, src.replace(".cu", ".o"))
            cmd = [nvcc()] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            return src, obj, r
        with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            results = list(ex.map(compile_one, SOURCES))
        for src, _, r in results:
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if not quiet and (r.stdout.strip() or r.stderr.strip()):
                print(r.stdout + r.stderr, file=sys.stderr)
        staged = os.path.join(tmp, "libssm.so")
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", staged] + [o for _, o, _ in results]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(staged, out)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return out


if __name__ == "__main__":
    path = build_library(force="--force" in sys.argv, verbose_ptxas="--ptxas-v" in sys.argv)
    print(path)
