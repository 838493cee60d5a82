"""Build the CUDA libraries in-tree for sm_103a.

    python -m selective_state_space_122_b300.build [--verbose]

* libssmscan.so -- the C-ABI selective-scan library (include/ssm_scan.h);
* libssmpeak.so -- the arithmetic-unit throughput probes the benchmark uses
  for its roofline denominators (not part of the scan path).

nvcc cross-compiles without a GPU.  Both libraries statically link the CUDA
runtime, so they only need the driver at run time.
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
PEAK_LIB = os.path.join(PKG, "libssmpeak.so")
PEAK_SOURCES = ["sfu_peak.cu"]
SOURCES = ["ssm_api.cu", "scan_fwd.cu", "scan_relay.cu", "scan_tmem.cu", "state_update.cu", "conv1d.cu", "scan_bwd.cu", "noalloc.cu"]
HEADERS = ["ssm_internal.cuh", "scan_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--shared", "-cudart", "static"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS]
            + [os.path.join(ROOT, "include", "ssm_scan.h")])


def up_to_date(out: str = LIB, inputs=None) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(p) <= t for p in (inputs or _inputs()))


def _nvcc(out: str, sources, verbose: bool) -> None:
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"),
           *(["-Xptxas", "-v"] if verbose else []),
           "-o", out, *[os.path.join(CSRC, s) for s in sources]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed building {os.path.basename(out)}")
    if verbose:
        sys.stderr.write(r.stderr)


def build(out: str = LIB, verbose: bool = False, force: bool = False) -> str:
    if force or not up_to_date(out):
        _nvcc(out, SOURCES, verbose)
    return out


def build_peak(out: str = PEAK_LIB, verbose: bool = False, force: bool = False) -> str:
    srcs = [os.path.join(CSRC, s) for s in PEAK_SOURCES]
    if force or not up_to_date(out, srcs):
        _nvcc(out, PEAK_SOURCES, verbose)
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/smem usage")
    ap.add_argument("--force", action="store_true")
    args = ap.parse_args()
    print(build(verbose=args.verbose, force=args.force or args.verbose))
    print(build_peak(verbose=args.verbose, force=args.force or args.verbose))
