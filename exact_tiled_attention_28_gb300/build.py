"""Builds libfa.so and libfa_debug.so in-tree from csrc/*.cu with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (all in parallel, the
release and the debug objects together), then one link step per library.
libfa_debug.so is the same sources with FA_DEBUG defined: its kernels check
their store indices and take their wait limit from a device variable (see
include/fa.h, "The debug build"). No CMake, no torch extension machinery.
Usage: ``python -m exact_tiled_attention_28_gb300.build [--verbose]``.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfa.so")
LIB_DEBUG = os.path.join(HERE, "libfa_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE]
VARIANTS = {"release": ([], LIB), "debug": (["-DFA_DEBUG=1"], LIB_DEBUG)}


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def _compile(src: str, variant: str, verbose: bool) -> tuple[str, str]:
    out_dir = os.path.join(BUILD, variant)
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *VARIANTS[variant][0], "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src} ({variant}):\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _link(objs: list, lib: str) -> None:
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(verbose: bool = False) -> str:
    """Builds both libraries; returns the path of the release one."""
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    jobs = [(s, v) for v in VARIANTS for s in srcs]
    for v in VARIANTS:
        os.makedirs(os.path.join(BUILD, v), exist_ok=True)
    workers = max(1, min(len(jobs), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        # the largest translation units first, so that they do not finish last
        jobs.sort(key=lambda j: -os.path.getsize(j[0]))
        results = dict(zip(jobs, ex.map(lambda j: _compile(j[0], j[1], verbose), jobs)))
    if verbose:
        for (s, v), (_, log) in sorted(results.items()):
            if v == "release":
                sys.stderr.write(log)
    for v, (_, lib) in VARIANTS.items():
        _link([results[(s, v)][0] for s in srcs], lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv))
