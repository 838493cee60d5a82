"""Build the CUDA libraries in-tree for sm_103a.

    python -m selective_state_space_122_b300.build [--verbose]

* libssmscan.so -- the C-ABI selective-scan library (include/ssm_scan.h);
* libssmpeak.so -- the arithmetic-unit throughput probes the benchmark uses
  for its roofline denominators (not part of the scan path).

nvcc cross-compiles without a GPU.  Both libraries statically link the CUDA
runtime, so they only need the NVIDIA GPU driver at run time.  The sources compile to
objects in parallel (under _build/ next to this file), then link once.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libssmscan.so")
PEAK_LIB = os.path.join(PKG, "libssmpeak.so")
PEAK_SOURCES = ["sfu_peak.cu"]
SOURCES = ["ssm_api.cu", "scan_fwd.cu", "scan_seg.cu", "scan_tmem.cu", "state_update.cu", "conv1d.cu", "scan_bwd.cu", "noalloc.cu"]
HEADERS = ["ssm_internal.cuh", "scan_common.cuh", "device_memo.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMPILE_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]
LINK_FLAGS = ["--shared", "-cudart", "static"]
OBJ_DIR = os.path.join(PKG, "_build")


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


def _run(cmd, what: str, verbose: bool) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed building {what}")
    if verbose:
        sys.stderr.write(r.stderr)


def _nvcc(out: str, sources, verbose: bool) -> None:
    """Compile every source to an object (in parallel), then link the shared library."""
    os.makedirs(OBJ_DIR, exist_ok=True)
    stem = os.path.splitext(os.path.basename(out))[0]
    objs = [os.path.join(OBJ_DIR, f"{stem}.{os.path.splitext(s)[0]}.o") for s in sources]

    def compile_one(src_obj):
        src, obj = src_obj
        _run([nvcc(), *ARCH, *COMPILE_FLAGS, "-I", os.path.join(ROOT, "include"),
              *(["-Xptxas", "-v"] if verbose else []), "-c", "-o", obj, os.path.join(CSRC, src)], src, verbose)

    workers = max(1, min(len(sources), os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as pool:
        list(pool.map(compile_one, zip(sources, objs)))
    _run([nvcc(), *ARCH, *LINK_FLAGS, "-o", out, *objs], os.path.basename(out), verbose)


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
