"""Build libmsc.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

    python -m selective_state_space_160_b300.build [--force] [--debug]

Objects go to _build/ under the package; the shared library lands next to this
file so that it travels with the source tree.
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmsc.so")
# Not part of the library: the tests' device fixtures (a one-CTA tcgen05 GEMM
# that checks the descriptors, a bounded wait that nothing completes) and the
# bench's pipe-throughput probe, each built into its own in-tree library.
FIXTURE_DIR = os.path.join(ROOT, "tests", "fixtures")
FIXTURE_LIB = os.path.join(FIXTURE_DIR, "libmsc_fixtures.so")
PIPE_PEAKS_SRC = os.path.join(ROOT, "bench_pipe_peaks.cu")
PIPE_PEAKS_LIB = os.path.join(ROOT, "libmsc_pipe_peaks.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _deps():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def build(force: bool = False, verbose: bool = False, extra=None) -> str:
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest = max(os.path.getmtime(p) for p in _deps())
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    objs = []
    flags = ARCH + NVCC_FLAGS + ["-I", INCLUDE, "-I", CSRC] + list(extra or [])
    for src in sources:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [nvcc()] + flags + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        objs.append(obj)
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def _build_side(srcs, lib, verbose=False, force=False):
    newest = max(os.path.getmtime(p) for p in srcs + _deps())
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return lib
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-cudart", "static",
                             "-I", INCLUDE, "-I", CSRC, "-o", tmp] + srcs
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def build_fixtures(force: bool = False, verbose: bool = False) -> str:
    """Build the tests' device fixtures (tests/fixtures/*.cu)."""
    return _build_side(sorted(glob.glob(os.path.join(FIXTURE_DIR, "*.cu"))), FIXTURE_LIB, verbose, force)


def build_pipe_peaks(force: bool = False, verbose: bool = False) -> str:
    """Build the bench's MUFU / FFMA throughput probe (bench_pipe_peaks.cu)."""
    return _build_side([PIPE_PEAKS_SRC], PIPE_PEAKS_LIB, verbose, force)


def build_all(force: bool = False, verbose: bool = False):
    return (build(force=force, verbose=verbose), build_fixtures(force=force, verbose=verbose),
            build_pipe_peaks(force=force, verbose=verbose))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print register / smem usage")
    args = ap.parse_args(argv)
    extra = ["-Xptxas", "-v"] if args.ptxas_info else None
    print(build(force=args.force or args.ptxas_info, verbose=args.verbose, extra=extra))
    print(build_fixtures(force=args.force, verbose=args.verbose))
    print(build_pipe_peaks(force=args.force, verbose=args.verbose))


if __name__ == "__main__":
    sys.exit(main())
