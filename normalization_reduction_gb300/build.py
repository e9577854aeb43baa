"""Builds libfnorm.so in-tree for GB300 (sm_103a) with nvcc.

Each CUDA translation unit under ``csrc/`` is compiled in parallel into
``_build/`` and the objects are linked into ``libfnorm.so`` beside this file.
Objects are rebuilt only when a source or header is newer than them.

    python -m normalization_reduction_gb300.build [--force] [--verbose] [--phases]
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


# Instrumented variant (build(phases=True), CLI --phases): the same sources
# with FNORM_PHASE_TRACE defined, which records per-phase %globaltimer stamps
# in the epilogue's L2-form kernel and exports fnorm_phase_trace_read; built
# into its own folder as libfnorm_phases.so for bench.py --phases. The product
# library never contains it.
BUILD_PHASES = os.path.join(HERE, "_build_phases")
LIBRARY_PHASES = os.path.join(HERE, "libfnorm_phases.so")


def _compile(src: str, verbose: bool, phases: bool = False) -> str:
    obj = os.path.join(BUILD_PHASES if phases else BUILD, os.path.splitext(src)[0] + ".o")
    extra = ["-DFNORM_PHASE_TRACE"] if phases else []
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, phases: bool = False) -> str:
    out_dir, library = (BUILD_PHASES, LIBRARY_PHASES) if phases else (BUILD, LIBRARY)
    os.makedirs(out_dir, exist_ok=True)
    newest = _deps_mtime()
    objs = [os.path.join(out_dir, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    todo = [s for s, o in zip(SOURCES, objs)
            if force or not os.path.exists(o) or os.path.getmtime(o) < newest]
    if todo:
        workers = min(len(todo), os.cpu_count() or 1)
        with cf.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(lambda s: _compile(s, verbose, phases), todo))
    if todo or not os.path.exists(library) or os.path.getmtime(library) < max(
            os.path.getmtime(o) for o in objs):
        tmp = library + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, library)
    return library


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--phases", action="store_true",
                    help="build the instrumented libfnorm_phases.so instead")
    a = ap.parse_args()
    print(build(a.force, a.verbose, a.phases))
