"""Builds libfnorm.so in-tree for GB300 (sm_103a) with nvcc.

Each CUDA translation unit under ``csrc/`` is compiled in parallel into
``_build/`` and the objects are linked into ``libfnorm.so`` beside this file.
Objects are rebuilt only when a source or header is newer than them.

    python -m normalization_reduction_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
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
LIBRARY = os.path.join(HERE, "libfnorm.so")
HEADER = os.path.join(ROOT, "include", "fnorm.h")
SOURCES = ["fnorm_api.cu", "in_f32.cu", "in_bf16.cu", "epi_kernels.cu", "bn_kernels.cu",
           "bn_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libfnorm")
    return exe


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*")) + [HEADER, os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    newest = _deps_mtime()
    objs = [os.path.join(BUILD, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    todo = [s for s, o in zip(SOURCES, objs)
            if force or not os.path.exists(o) or os.path.getmtime(o) < newest]
    if todo:
        workers = min(len(todo), os.cpu_count() or 1)
        with cf.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(lambda s: _compile(s, verbose), todo))
    if todo or not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < max(
            os.path.getmtime(o) for o in objs):
        tmp = LIBRARY + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(a.force, a.verbose))
