"""Profiling drivers for the selective-scan library (run on a CUDA device).

    python -m selective_state_space_122_b300.profile scan [--batch B] [--dim D] [--L L]
           [--N N] [--iters K] [--path tmem2|ws|seg|generic] [--ngroups G]
    python -m selective_state_space_122_b300.profile decode [--batch B] [--dim D] [--N N] [--iters K] [--ngroups G]
           [--graph STEPS]
    python -m selective_state_space_122_b300.profile conv [--batch B] [--dim D] [--L L] [--W W] [--iters K]
    python -m selective_state_space_122_b300.profile bwd [--batch B] [--dim D] [--L L] [--N N] [--iters K] [--ngroups G]
    python -m selective_state_space_122_b300.profile units

``scan`` runs ssm_scan_fwd on seeded on-device bf16 inputs shaped like the
pages' workloads (u, delta_raw, z, B, C ~ N(0, 1); A = -(1..N); D = 1;
delta_bias = softplus^-1(dt), dt log-uniform in [1e-3, 0.1]) and prints the
CUDA-event time of each call: the command behind the ncu captures of the scan
kernels.  ``decode`` does the same for one ssm_state_update step; with
``--graph STEPS`` it also times STEPS back-to-back steps issued eagerly against
the same steps captured once into a CUDA graph and replayed (per step).  --ngroups
draws B and C per channel group (the grouped entry points).  ``units``
prints the measured SFU (ex2, tanh) and packed-FMA throughput at 1, 2 and 8
warps per scheduler, and the ex2 rate when each ex2 is followed by 0, 1 or 2
independent packed FMAs -- the SFU / FMA-pipe mix of a recurrence step --
and the rate of the in-warp time-split core (16 states per lane over short
sub-chunks, warp-shuffle combine, re-sweep) with the long-sequence scan time
it implies (libssmpeak.so).
"""
from __future__ import annotations

import argparse
import ctypes
import math
import os
import sys

import torch

from . import build as libbuild
from ._lib import device_error, force_scan_path, scan_workspace_bytes, ssm_scan_fwd, ssm_state_update


def _inputs(batch, dim, L, N, dev, seed=0, ngroups=1):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    u = torch.randn(batch, L, dim, device=dev, generator=g).bfloat16()
    dl = torch.randn(batch, L, dim, device=dev, generator=g).bfloat16()
    z = torch.randn(batch, L, dim, device=dev, generator=g).bfloat16()
    bc = (batch, N, L) if ngroups == 1 else (batch, ngroups, N, L)
    B = torch.randn(*bc, device=dev, generator=g).bfloat16()
    C = torch.randn(*bc, device=dev, generator=g).bfloat16()
    A = -torch.arange(1, N + 1, device=dev, dtype=torch.float32).repeat(dim, 1).contiguous()
    D = torch.ones(dim, device=dev)
    dt = torch.exp(torch.empty(dim, device=dev).uniform_(math.log(1e-3), math.log(0.1), generator=g))
    bias = dt + torch.log(-torch.expm1(-dt))
    return u, dl, z, B, C, A, D, bias


def cmd_scan(a):
    if a.path:
        force_scan_path(a.path)
    dev = torch.device("cuda", 0)
    u, dl, z, B, C, A, D, bias = _inputs(a.batch, a.dim, a.L, a.N, dev, ngroups=a.ngroups)
    out = torch.empty_like(u)
    last = torch.empty(a.batch, a.dim, a.N, device=dev)
    ws = torch.empty(max(16, scan_workspace_bytes(a.batch, a.dim, a.L, a.N, torch.bfloat16, a.ngroups)),
                     dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    elems = a.batch * a.dim * a.L * a.N
    for i in range(a.iters):
        e0.record()
        ssm_scan_fwd(u, dl, A, B, C, D, z, bias, True, out=out, last_state=last, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"scan {a.batch}x{a.dim}x{a.L} N{a.N} G{a.ngroups} iter {i}: {ms:.3f} ms "
              f"({elems / (ms * 1e-3) / 1e9:.1f} G elements/s)", flush=True)
    err = device_error()
    print("device error word:", err)
    return 0 if err == 0 else 1


def cmd_decode(a):
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    st = torch.randn(a.batch, a.dim, a.N, device=dev, generator=g) * 0.1
    x, dt, z = (torch.randn(a.batch, a.dim, device=dev, generator=g).bfloat16() for _ in range(3))
    bc = (a.batch, a.N) if a.ngroups == 1 else (a.batch, a.ngroups, a.N)
    B, C = (torch.randn(*bc, device=dev, generator=g).bfloat16() for _ in range(2))
    A = -torch.arange(1, a.N + 1, device=dev, dtype=torch.float32).repeat(a.dim, 1).contiguous()
    D = torch.ones(a.dim, device=dev)
    bias = torch.full((a.dim,), -4.0, device=dev)
    out = torch.empty_like(x)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nbytes = 2 * st.numel() * 4 + 4 * x.numel() * 2
    for i in range(a.iters):
        e0.record()
        ssm_state_update(st, x, dt, A, B, C, D, z, bias, True, out=out)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"decode {a.batch}x{a.dim} N{a.N} G{a.ngroups} iter {i}: {ms * 1e3:.1f} us "
              f"({nbytes / (ms * 1e-3) / 1e9:.0f} GB/s)", flush=True)
    if a.graph:
        def steps():
            for _ in range(a.graph):
                ssm_state_update(st, x, dt, A, B, C, D, z, bias, True, out=out)

        def per_step(fn):
            best = float("inf")
            for _ in range(5):
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1) / a.graph)
            return best

        eager = per_step(steps)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            steps()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            steps()
        graph = per_step(g.replay)
        print(f"decode {a.batch}x{a.dim} N{a.N}: {a.graph} steps, eager {eager * 1e3:.2f} us/step, "
              f"CUDA graph replay {graph * 1e3:.2f} us/step", flush=True)
    return 0


def cmd_bwd(a):
    from ._lib import ssm_scan_bwd
    dev = torch.device("cuda", 0)
    u, dl, z, B, C, A, D, bias = _inputs(a.batch, a.dim, a.L, a.N, dev, ngroups=a.ngroups)
    dout = torch.randn_like(u, dtype=torch.float32).bfloat16()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    elems = a.batch * a.dim * a.L * a.N
    ws = None
    for i in range(a.iters):
        e0.record()
        ssm_scan_bwd(u, dl, A, B, C, D, z, bias, True, dout, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"bwd {a.batch}x{a.dim}x{a.L} N{a.N} G{a.ngroups} iter {i}: {ms:.3f} ms "
              f"({elems / (ms * 1e-3) / 1e9:.1f} G elements/s)", flush=True)
    return 0


def cmd_conv(a):
    from ._lib import conv1d_fwd
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(2)
    x = torch.randn(a.batch, a.L, a.dim, device=dev, generator=g).bfloat16()
    w = torch.randn(a.dim, a.W, device=dev, generator=g) * 0.5
    bias = torch.randn(a.dim, device=dev, generator=g) * 0.5
    st = torch.zeros(a.batch, a.dim, a.W - 1, device=dev)
    out = torch.empty_like(x)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nbytes = 2 * x.numel() * 2
    for i in range(a.iters):
        e0.record()
        conv1d_fwd(x, w, bias, True, st, out=out, state_out=st)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"conv {a.batch}x{a.L}x{a.dim} W{a.W} iter {i}: {ms:.3f} ms "
              f"({nbytes / (ms * 1e-3) / 1e9:.0f} GB/s)", flush=True)
    return 0


def cmd_units(a):
    lib = ctypes.CDLL(libbuild.PEAK_LIB)
    lib.ssmpk_probe_shape.argtypes = [ctypes.c_int] * 4
    lib.ssmpk_probe_shape.restype = ctypes.c_double
    lib.ssmpk_sm_count.restype = ctypes.c_int
    sms = lib.ssmpk_sm_count()
    for name, kind, iters in (("ex2", 0, 20000), ("packed FMA", 3, 40000), ("tanh", 4, 10000)):
        for bps, thr in ((1, 128), (2, 128), (4, 256)):
            r = max(lib.ssmpk_probe_shape(kind, iters, bps, thr) for _ in range(3))
            wps = bps * thr // 32 / 4
            print(f"{name:10s} {wps:3.0f} warp(s)/scheduler: {r / 1e9:9.1f} G/s "
                  f"= {r / (sms * a.clock_mhz * 1e6):6.2f} per clock per SM (at {a.clock_mhz:.0f} MHz)")
    # co-issue: ex2 alone, then each ex2 followed by 1 or 2 independent packed FMAs
    for name, kind in (("ex2 + 0 FFMA2", 5), ("ex2 + 1 FFMA2", 6), ("ex2 + 2 FFMA2", 7)):
        for bps, thr in ((1, 128), (4, 256)):
            r = max(lib.ssmpk_probe_shape(kind, 20000, bps, thr) for _ in range(3))
            wps = bps * thr // 32 / 4
            per = r / (sms * a.clock_mhz * 1e6)
            print(f"{name:14s} {wps:3.0f} warp(s)/scheduler: {per:6.2f} ex2 per clock per SM "
                  f"({128.0 / per:5.2f} cycles per warp-wide ex2 on a scheduler)")
    # the in-warp time-split core (16 states per lane over T-step sub-chunks,
    # shuffle combine, re-sweep) and what it implies for the long-sequence
    # scan's 1 x 5120 x 131072 x 16 elements
    lib.ssmpk_timesplit.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.ssmpk_timesplit.restype = ctypes.c_double
    elems = 5120 * 131072 * 16
    for T in (2, 4):
        r = max(lib.ssmpk_timesplit(T, 2000) for _ in range(3))
        print(f"time-split core T={T}: {r / 1e9:8.1f} G elements/s = {r / (sms * a.clock_mhz * 1e6):6.2f} "
              f"per clock per SM; the long-sequence scan's elements alone: {elems / r * 1e3:6.3f} ms")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    sub = ap.add_subparsers(dest="cmd", required=True)
    s = sub.add_parser("scan")
    s.add_argument("--batch", type=int, default=1)
    s.add_argument("--dim", type=int, default=5120)
    s.add_argument("--L", type=int, default=16384)
    s.add_argument("--N", type=int, default=16)
    s.add_argument("--iters", type=int, default=3)
    s.add_argument("--path", default=None, choices=[None, "tmem2", "ws", "seg", "generic"])
    s.add_argument("--ngroups", type=int, default=1)
    d = sub.add_parser("decode")
    d.add_argument("--batch", type=int, default=256)
    d.add_argument("--dim", type=int, default=5120)
    d.add_argument("--N", type=int, default=16)
    d.add_argument("--iters", type=int, default=5)
    d.add_argument("--ngroups", type=int, default=1)
    d.add_argument("--graph", type=int, default=0, help="also time this many steps eagerly and as a CUDA graph")
    bw = sub.add_parser("bwd")
    bw.add_argument("--batch", type=int, default=8)
    bw.add_argument("--dim", type=int, default=2048)
    bw.add_argument("--L", type=int, default=2048)
    bw.add_argument("--N", type=int, default=16)
    bw.add_argument("--iters", type=int, default=3)
    bw.add_argument("--ngroups", type=int, default=1)
    cv = sub.add_parser("conv")
    cv.add_argument("--batch", type=int, default=1)
    cv.add_argument("--dim", type=int, default=5120)
    cv.add_argument("--L", type=int, default=131072)
    cv.add_argument("--W", type=int, default=4)
    cv.add_argument("--iters", type=int, default=5)
    u = sub.add_parser("units")
    u.add_argument("--clock-mhz", type=float, default=2032.0)
    a = ap.parse_args(argv)
    return {"scan": cmd_scan, "decode": cmd_decode, "conv": cmd_conv, "bwd": cmd_bwd, "units": cmd_units}[a.cmd](a)


if __name__ == "__main__":
    sys.exit(main())
