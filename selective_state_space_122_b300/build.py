"""Build libssmscan.so (the C-ABI CUDA library) in-tree for sm_103a.

    python -m selective_state_space_122_b300.build [--verbose]

nvcc cross-compiles without a GPU.  The library statically links the CUDA
runtime, so it only needs the driver at run time.
"""
from __future__ import annotations

import argparse
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libssmscan.so")
SOURCES = ["ssm_api.cu", "scan_fwd.cu", "state_update.cu"]
HEADERS = ["ssm_internal.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--shared", "-cudart", "static"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS]
            + [os.path.join(ROOT, "include", "ssm_scan.h")])


def up_to_date(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(out: str = LIB, verbose: bool = False, force: bool = False) -> str:
    if not force and up_to_date(out):
        return out
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"),
           *(["-Xptxas", "-v"] if verbose else []),
           "-o", out, *[os.path.join(CSRC, s) for s in SOURCES]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed building libssmscan.so")
    if verbose:
        sys.stderr.write(r.stderr)
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/smem usage")
    ap.add_argument("--force", action="store_true")
    args = ap.parse_args()
    print(build(verbose=args.verbose, force=args.force or args.verbose))
