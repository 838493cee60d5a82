"""Benchmark of the selective-scan hot path on one (or N replica) B300s.

One step = one full-sequence selective scan over the long-sequence workload
(batch 1, d_inner 5120, L 131072, d_state 16, bf16 activations) followed by
one recurrent decode step over the batched decode workload (batch 256,
d_inner 5120, d_state 16, fp32 state updated in place).  Both run through the
library's C ABI on inputs resident in HBM; the scan's 5.4 GB of traffic per
step is far larger than the 126 MB L2, so no explicit flush is needed between
steps and the decode state (84 MB) is evicted by the scan that precedes it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Under torchrun every rank runs an independent
replica (the path has no data exchange); time is the max over ranks.

``--impl reference`` times the float64 CPU oracle on the host cores on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_122_b300 import inputs  # noqa: E402

METRIC = "selective-scan elements (B·D·L·N)/s and achieved HBM GB/s vs roofline, 1 B300"
SCAN = inputs.LONG_SEQ
DECODE = inputs.DECODE_256
# Special-function work of the method per (b, t, d), in exp2-equivalents: N
# exp2 for exp(Delta A), plus 4 for softplus (exp2 + log) and silu (exp2 +
# reciprocal) -- the (N + 4) unit the roofline is quoted in, against the
# exp2 rate measured on the GPU by libssmpeak.so before the timed region.
def sfu_units_per_td(n):
    return n + 4


# What the benchmarked kernel actually issues per (b, t, d): N + 1 exp2
# (decays and softplus, whose log1p is a polynomial on the FMA pipe) and one
# tanh (silu(z) = (z/2)(1 + tanh(z/2))).
def sfu_issued_per_td(n):
    return {"ex2": n + 1, "tanh": 1}


FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "sm_max_mhz": 2032.0, "source": "fallback"}


# ---------------------------------------------------------------- accounting

def scan_elements(s=SCAN):
    return s.batch * s.dim * s.seqlen * s.dstate


# dram__bytes_read.sum + dram__bytes_write.sum of scan_tmem2_kernel as built
# (conflict-free shared-memory layouts), from one ncu capture of the
# long-sequence workload cut to L = 16384
# (profiles/scan_tmem2_kernel_1x5120x16384.md), scaled by 131072 / 16384: the
# traffic grows in proportion to L.
SCAN_TRAFFIC_L16384 = 654.7e6
SCAN_TRAFFIC_BYTES = SCAN_TRAFFIC_L16384 * 8


def scan_bytes(s=SCAN, es=2):
    """Algorithmic HBM bytes of one scan: u, delta, z read and out written once
    per (b, t, d); B and C once; A, D, delta_bias once; final state written."""
    btd = s.batch * s.seqlen * s.dim
    return (4 * btd * es + 2 * s.batch * s.dstate * s.seqlen * es
            + s.dim * s.dstate * 4 + 2 * s.dim * 4 + s.batch * s.dim * s.dstate * 4)


def scan_sfu_units(s=SCAN):
    """SFU work of one scan in the roofline's unit: (N + 4) exp2-equivalents per (b, t, d)."""
    return s.batch * s.seqlen * s.dim * sfu_units_per_td(s.dstate)


def scan_sfu_issued_seconds(rates, s=SCAN):
    """Time the SFU needs for the instructions the kernel issues, at the measured rates."""
    btd = s.batch * s.seqlen * s.dim
    return sum(btd * k / rates[op] for op, k in sfu_issued_per_td(s.dstate).items())


def decode_elements(s=DECODE):
    return s.batch * s.dim * s.dstate


def decode_bytes(s=DECODE, es=2):
    """State read + written (fp32), x, dt, z read and out written, B, C, A, D, bias."""
    return (2 * s.batch * s.dim * s.dstate * 4 + 4 * s.batch * s.dim * es
            + 2 * s.batch * s.dstate * es + s.dim * s.dstate * 4 + 2 * s.dim * 4)


def probe_units(device_index=0):
    """Throughput of the special-function unit (ex2, lg2, rcp) and of packed
    float32 FMA on this GPU, measured by libssmpeak.so (ops/s)."""
    import ctypes
    from selective_state_space_122_b300 import build as libbuild
    path = libbuild.PEAK_LIB
    if not os.path.exists(path):
        return None
    lib = ctypes.CDLL(path)
    lib.ssmpk_probe.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.ssmpk_probe.restype = ctypes.c_double
    lib.ssmpk_sm_count.restype = ctypes.c_int
    out = {}
    for name, kind, iters in (("ex2", 0, 20000), ("lg2", 1, 10000), ("rcp", 2, 10000), ("ffma", 3, 40000),
                              ("tanh", 4, 10000)):
        best = max(lib.ssmpk_probe(kind, iters, 4) for _ in range(3))
        out[name] = best
    out["sms"] = lib.ssmpk_sm_count()
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "sm_max_mhz": float(d.get("sm_max_mhz", 2032.0)),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS)


# ---------------------------------------------------------------- distributed

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value, world, device=None):
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 50 ms while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        # the samples are also kept as a file: SSM_BENCH_CLOCK_DIR, else the temp directory
        out_dir = os.environ.get("SSM_BENCH_CLOCK_DIR") or tempfile.gettempdir()
        os.makedirs(out_dir, exist_ok=True)
        self.path = os.path.join(out_dir, f"clocks_rank{self.gpu}.csv")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        return summarize_clock_samples(open(self.path).read().splitlines())


def summarize_clock_samples(lines):
    """Clock record of the timed region from nvidia-smi CSV rows (the QUERY
    fields, no header, no units): the median SM clock over the samples under
    load (drawing at least half the peak power seen; the sampler also runs a
    moment before and after the timed region), the maximum clock, and every
    throttle reason seen active.  A row whose power reads as unavailable still
    counts for the clocks and the reasons."""
    sm, smax, power, reasons = [], [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            c, cm = float(f[1]), float(f[2])
        except ValueError:
            continue
        try:
            w = float(f[3])
        except ValueError:
            w = None
        sm.append(c)
        smax.append(cm)
        power.append(w)
        for n, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    known = [w for w in power if w is not None]
    pk = max(known) if known else None
    loaded = [c for c, w in zip(sm, power) if w is not None and w >= 0.5 * pk] if known else []
    loaded = loaded or sm
    return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "samples": len(sm),
            "samples_under_load": len(loaded), "power_w_max": pk, "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our arm

def make_workload(device):
    """Seeded inputs generated on the host and made resident on the device."""
    import torch

    def up(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)

    si = inputs.make_scan_inputs(SCAN, 3)
    di = inputs.make_decode_inputs(DECODE, 4)
    x, dt, z, B, C = di.token()
    w = {
        "scan_host": si,
        "scan": {k: up(getattr(si, k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias")},
        "dec": {"state": up(di.state0), "x": up(x), "dt": up(dt), "z": up(z), "B": up(B), "C": up(C),
                "A": up(di.A), "D": up(di.D), "dt_bias": up(di.dt_bias)},
        "dec_host": (di, x, dt, z, B, C),
    }
    s = w["scan"]
    from selective_state_space_122_b300 import scan_workspace_bytes
    w["ws"] = torch.empty(scan_workspace_bytes(SCAN.batch, SCAN.dim, SCAN.seqlen, SCAN.dstate, torch.bfloat16),
                          dtype=torch.uint8, device=device)
    w["scan_out"] = torch.empty_like(s["u"])
    w["scan_last"] = torch.empty((SCAN.batch, SCAN.dim, SCAN.dstate), dtype=torch.float32, device=device)
    w["dec_out"] = torch.empty_like(w["dec"]["x"])
    return w


def run_step(w, ev=None):
    """One step of the hot path: the long-sequence scan, then one decode step."""
    from selective_state_space_122_b300 import ssm_scan_fwd, ssm_state_update
    s, d = w["scan"], w["dec"]
    if ev is not None:
        ev[0].record()
    ssm_scan_fwd(s["u"], s["delta"], s["A"], s["B"], s["C"], s["D"], s["z"], s["delta_bias"], True,
                 out=w["scan_out"], last_state=w["scan_last"], workspace=w["ws"])
    if ev is not None:
        ev[1].record()
    ssm_state_update(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                     True, out=w["dec_out"])
    if ev is not None:
        ev[2].record()


def run_e2e(w, steps, device, pieces=16):
    """The same step through the public API from pinned HOST buffers: every
    input of the step is copied host->device and both outputs device->host,
    inside the timed region.  The long sequence is streamed in ``pieces``
    consecutive pieces, as a user with the data on the host would: piece k+1
    is copied in on one stream while piece k is scanned on another, starting
    from the state piece k-1 left (ssm_scan_fwd with initial_state), and piece
    k-1's output is copied back on a third; the decode step follows.  Same
    bytes moved as one whole-step copy, same results."""
    import torch
    from selective_state_space_122_b300 import ssm_scan_fwd, ssm_state_update
    s, d = w["scan"], w["dec"]
    hs = {k: v.cpu().pin_memory() for k, v in s.items()}
    hd = {k: v.cpu().pin_memory() for k, v in d.items()}
    out_h = torch.empty(w["scan_out"].shape, dtype=w["scan_out"].dtype).pin_memory()
    last_h = torch.empty(w["scan_last"].shape, dtype=torch.float32).pin_memory()
    dec_out_h = torch.empty(w["dec_out"].shape, dtype=w["dec_out"].dtype).pin_memory()
    dec_state_h = torch.empty(d["state"].shape, dtype=torch.float32).pin_memory()
    ds = {k: torch.empty_like(v) for k, v in s.items()}
    dd = {k: torch.empty_like(v) for k, v in d.items()}
    h2d = sum(v.numel() * v.element_size() for v in hs.values()) + \
        sum(v.numel() * v.element_size() for v in hd.values())
    d2h = (out_h.numel() * out_h.element_size() + last_h.numel() * 4
           + dec_out_h.numel() * dec_out_h.element_size() + dec_state_h.numel() * 4)
    bt, L, _ = s["u"].shape
    N = s["B"].shape[1]
    if bt > 1:
        pieces = 1        # (batch, L, dim) pieces of more than one row are not contiguous
    step_len = ((L + pieces - 1) // pieces + 63) // 64 * 64
    bounds = [(lo, min(lo + step_len, L)) for lo in range(0, L, step_len)]
    # B and C pieces are (batch, N, piece) rows of the (batch, N, L) arrays: two
    # contiguous device buffers, alternating between pieces
    bc_buf = [[torch.empty((bt, N, step_len), dtype=s["B"].dtype, device=device) for _ in range(2)]
              for _ in range(2)]
    copy_in, copy_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    compute = torch.cuda.current_stream(device)
    state = w["scan_last"]

    def one():
        done = []
        with torch.cuda.stream(copy_in):
            copy_in.wait_stream(compute)
            for k in ("A", "D", "delta_bias"):
                ds[k].copy_(hs[k], non_blocking=True)
        for i, (lo, hi) in enumerate(bounds):
            n = hi - lo
            Bp, Cp = bc_buf[0][i % 2], bc_buf[1][i % 2]
            with torch.cuda.stream(copy_in):
                if i >= 2:
                    copy_in.wait_event(done[i - 2])      # the B/C buffer is free again
                for k in ("u", "delta", "z"):
                    ds[k][:, lo:hi].copy_(hs[k][:, lo:hi], non_blocking=True)
                for b in range(bt):
                    for r in range(N):
                        Bp[b, r, :n].copy_(hs["B"][b, r, lo:hi], non_blocking=True)
                        Cp[b, r, :n].copy_(hs["C"][b, r, lo:hi], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(copy_in)
            compute.wait_event(ready)
            ssm_scan_fwd(ds["u"][:, lo:hi], ds["delta"][:, lo:hi], ds["A"], Bp[:, :, :n].contiguous()
                         if n != step_len else Bp, Cp[:, :, :n].contiguous() if n != step_len else Cp,
                         ds["D"], ds["z"][:, lo:hi], ds["delta_bias"], True, out=w["scan_out"][:, lo:hi],
                         last_state=state, initial_state=None if i == 0 else state, workspace=w["ws"])
            ev = torch.cuda.Event()
            ev.record(compute)
            done.append(ev)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(ev)
                out_h[:, lo:hi].copy_(w["scan_out"][:, lo:hi], non_blocking=True)
        with torch.cuda.stream(copy_in):
            for k in dd:
                dd[k].copy_(hd[k], non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(copy_in)
        compute.wait_event(ready)
        y = ssm_state_update(dd["state"], dd["x"], dd["dt"], dd["A"], dd["B"], dd["C"], dd["D"], dd["z"],
                             dd["dt_bias"], True, out=w["dec_out"])
        ev = torch.cuda.Event()
        ev.record(compute)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(ev)
            last_h.copy_(state, non_blocking=True)
            dec_out_h.copy_(y, non_blocking=True)
            dec_state_h.copy_(dd["state"], non_blocking=True)
        compute.wait_stream(copy_out)
        compute.wait_stream(copy_in)

    one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    for _ in range(steps):
        one()
    e1.record(compute)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # the streamed result equals the one-call scan on device-resident inputs
    run_step(w)
    torch.cuda.synchronize()
    same = bool(torch.equal(out_h, w["scan_out"].cpu())) and bool(torch.equal(last_h, w["scan_last"].cpu()))
    return ms, h2d, d2h, same


def time_side_kernels(w, device, iters=5):
    """CUDA-event times, outside the timed step, of:
    * the backward of the scan at the mid-size prefill shape (8 x 2048 x 2048,
      N 16, bf16; every input's gradient);
    * the causal conv1d + SiLU over the long-sequence activations (1 x 131072
      x 5120, width 4, bf16);
    * the decode step alone, each launch after a read of 512 MB that leaves
      the L2 clean (in the step it runs after the scan, whose output lines are
      still dirty in L2 and are written back during the decode); the mean of
      40 launches, since one ~30 us launch is only a few ticks of the event
      timer (2.05 us on this hardware).
    Inputs: seeded, on the device."""
    import torch
    from selective_state_space_122_b300 import conv1d_fwd, ssm_scan_bwd, ssm_state_update
    res = {}
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn, before=None, n=iters, reduce=statistics.median):
        ts = []
        for i in range(n + 2):
            if before is not None:
                before()
            e0, e1 = ev(), ev()
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if i >= 2:
                ts.append(e0.elapsed_time(e1))
        return reduce(ts)

    g = torch.Generator(device=device)
    g.manual_seed(5)
    bt, dim, L, N = 8, 2048, 2048, 16
    u, dl, z, dout = (torch.randn(bt, L, dim, device=device, generator=g).bfloat16() for _ in range(4))
    B, C = (torch.randn(bt, N, L, device=device, generator=g).bfloat16() for _ in range(2))
    A = -torch.arange(1, N + 1, device=device, dtype=torch.float32).repeat(dim, 1).contiguous()
    D = torch.ones(dim, device=device)
    dt = torch.exp(torch.empty(dim, device=device).uniform_(np.log(1e-3), np.log(0.1), generator=g))
    bias = dt + torch.log(-torch.expm1(-dt))
    res["bwd_ms"] = timed(lambda: ssm_scan_bwd(u, dl, A, B, C, D, z, bias, True, dout))
    del u, dl, z, dout, B, C
    s = w["scan"]
    wt = torch.randn(SCAN.dim, 4, device=device, generator=g) * 0.5
    cb = torch.randn(SCAN.dim, device=device, generator=g) * 0.1
    res["conv_ms"] = timed(lambda: conv1d_fwd(s["u"], wt, cb, True, out=w["scan_out"]))
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    flush.zero_()
    d = w["dec"]
    res["decode_isolated_us"] = 1e3 * timed(
        lambda: ssm_state_update(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                 d["dt_bias"], True, out=w["dec_out"]),
        before=lambda: flush.view(torch.int64).sum(), n=40, reduce=statistics.mean)
    torch.cuda.synchronize()
    return res


def cpu_baseline_sample(si, target_s=12.0, max_channels=None):
    """Time the float64 oracle (as it stands) on a bounded channel sample of the
    long-sequence scan ``si``, all host cores.  Returns a dict for the JSON line."""
    import oracle
    threads = oracle.max_threads()

    def run(ch):
        g = si.channels(np.arange(ch)).as_f64()
        t0 = time.perf_counter()
        oracle.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"], True)
        return time.perf_counter() - t0

    ch = max(threads, 8)
    dt = run(ch)
    want = int(ch * target_s / max(dt, 1e-3))
    want = max(ch, min(want, max_channels or SCAN.dim, SCAN.dim))
    want = max(threads, (want // threads) * threads) if want >= threads else want
    dt = run(want)
    elems = want * SCAN.seqlen * SCAN.dstate
    return {"value": elems / dt, "unit": "elements/s", "cores": threads, "kind": "oracle",
            "sample": f"{want} of 5120 channels x {SCAN.seqlen} steps x {SCAN.dstate} states "
                      f"(long-sequence scan), float64, {dt:.1f} s wall"}


def bench_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    from selective_state_space_122_b300 import load_library
    load_library()
    units = probe_units(local)
    clocks_mhz_for_units = load_peaks()["sm_max_mhz"]   # per-clock figures are at the maximum SM clock
    w = make_workload(device)
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        run_step(w)
    torch.cuda.synchronize()
    barrier(world)

    stream = torch.cuda.current_stream(device)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e_start.record(stream)
        for k in range(args.steps):
            run_step(w, evs[k])
        e_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    total_ms = e_start.elapsed_time(e_end)
    scan_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms = max_over_ranks(total_ms, world, device)
    clocks = clk.summary()

    side = time_side_kernels(w, device)

    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h, same = run_e2e(w, args.e2e_steps, device)
        e2e_ms = max_over_ranks(e2e_ms, world, device)
        e2e = (e2e_ms, h2d, d2h, same)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(w["scan_host"], args.cpu_seconds)

    if rank != 0:
        barrier(world)
        return None

    peaks = load_peaks()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    ms_step = total_ms / args.steps
    elems = (scan_elements() + decode_elements()) * world
    scan_avg = statistics.mean(scan_ms)
    dec_avg = statistics.mean(dec_ms)
    sfu_units = scan_sfu_units()
    t_sfu = sfu_units / units["ex2"]
    t_hbm = scan_bytes() / (peaks["hbm_gbs"] * 1e9)
    sfu_ach = sfu_units / (scan_avg * 1e-3)
    hbm_ach = scan_bytes() / (scan_avg * 1e-3) / 1e9
    t_roof_ms = max(t_hbm, t_sfu) * 1e3
    t_issued = scan_sfu_issued_seconds(units)
    dec_iso = side["decode_isolated_us"]
    line = {
        "metric": METRIC,
        "value": elems / (ms_step * 1e-3),
        "unit": "elements/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": ("long-sequence scan 1x5120x131072 d_state 16 (bf16 u/delta/z/B/C, f32 A/D/bias, "
                         "final state) + one decode step 256x5120 d_state 16 (f32 state in place)"),
            "io_dtype": "bf16",
            "l2": "no flush: each step streams 5.4 GB (> 126 MB L2) before the decode step",
            "parallelism": f"replicas x{world}",
            "sms": sms,
        },
        "scan_ms": scan_avg,
        "decode_us": dec_avg * 1e3,
        "bwd_ms": side["bwd_ms"],
        "conv_ms": side["conv_ms"],
        "roofline": {
            "bound": "alu",
            "unit": "G ex2-equiv/s",
            "achieved": sfu_ach / 1e9,
            "peak": units["ex2"] / 1e9,
            "frac": sfu_ach / units["ex2"],
            "traffic": SCAN_TRAFFIC_BYTES,
            "traffic_source": "ncu dram bytes of scan_tmem2_kernel (as built) at L=16384, x 8",
            "kernel": "ssm_scan_fwd: tm2_stage_kernel + scan_tmem2_kernel (long-sequence scan)",
            "work_unit": "(N + 4) exp2-equivalents per (b, t, d): N decays, softplus, silu",
            "peak_source": ("measured on this GPU by libssmpeak.so: ex2 %.1f, lg2 %.1f, rcp %.1f, tanh %.1f G/s, "
                            "packed FMA %.1f TFLOP/s"
                            % (units["ex2"] / 1e9, units["lg2"] / 1e9, units["rcp"] / 1e9, units["tanh"] / 1e9,
                               2 * units["ffma"] / 1e12)),
            "sfu_units_per_launch": sfu_units,
            "issued_sfu_per_td": sfu_issued_per_td(SCAN.dstate),
            "frac_issued": t_issued / (scan_avg * 1e-3),
            "sfu_per_sm_per_clk": {k: units[k] / (sms * clocks_mhz_for_units * 1e6)
                                   for k in ("ex2", "lg2", "rcp", "tanh", "ffma")},
            "hbm": {"achieved_gbs": hbm_ach, "peak_gbs": peaks["hbm_gbs"],
                    "frac": hbm_ach / peaks["hbm_gbs"], "bytes_per_launch": scan_bytes(),
                    "peak_source": peaks["source"]},
            "t_sfu_ms": t_sfu * 1e3,
            "t_hbm_ms": t_hbm * 1e3,
            # diagnostic: the float32 pipe's share, 4 FMA-pipe operations per
            # element (Delta A, Delta u B, the state FMA, C . h) at the
            # measured packed-FMA rate
            "t_fma_ms": 4 * scan_elements() / units["ffma"] * 1e3,
            "t_roof_ms": t_roof_ms,
            "frac_of_roofline_time": t_roof_ms / scan_avg,
        },
        "decode": {
            "us_per_step": dec_avg * 1e3,
            "bytes_per_step": decode_bytes(),
            "achieved_gbs": decode_bytes() / (dec_avg * 1e-3) / 1e9,
            "frac_hbm_in_step": decode_bytes() / (dec_avg * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "isolated_us": dec_iso,
            "frac_hbm": decode_bytes() / (dec_iso * 1e-6) / 1e9 / peaks["hbm_gbs"],
            "note": ("frac_hbm: the step alone after a clean L2; in the step it follows the scan, whose "
                     "dirty output lines in L2 are written back during it"),
        },
        "side_kernels": {
            "bwd": {"workload": "backward 8x2048x2048 d_state 16 bf16 (every gradient)", "ms": side["bwd_ms"]},
            "conv1d": {"workload": "causal conv1d + SiLU 1x131072x5120 width 4 bf16", "ms": side["conv_ms"],
                       "achieved_gbs": 2 * SCAN.batch * SCAN.seqlen * SCAN.dim * 2 / (side["conv_ms"] * 1e-3) / 1e9},
        },
        "clocks": clocks,
        "gpu_launches": 3 * args.steps,
    }
    if e2e is not None:
        e2e_ms, h2d, d2h, same = e2e
        line["e2e"] = {"value": elems / (e2e_ms * 1e-3), "unit": "elements/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                       "steps": args.e2e_steps,
                       "method": "sequence streamed in 16 pieces: copy-in, scan from the carried state "
                                 "and copy-out overlapped on three streams",
                       "output_equals_device_resident_scan": same}
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    barrier(world)
    return line


# ---------------------------------------------------------------- reference arm

def bench_reference(args):
    """The float64 oracle timed on the host cores: each step is a bounded
    channel sample of the long-sequence scan."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.load()
    threads = oracle.max_threads()
    ch = max(threads, args.ref_channels)
    si = inputs.make_scan_inputs(SCAN, 3)
    g = si.channels(np.arange(ch)).as_f64()
    del si

    def step():
        oracle.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"], True)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    elems = ch * SCAN.seqlen * SCAN.dstate
    value = elems / dt
    line = {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "elements/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": ("long-sequence scan 1x5120x131072 d_state 16: float64 CPU oracle on a "
                                f"{ch}-channel sample per step"), "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "elements/s", "cores": threads, "kind": "oracle",
                         "sample": f"{ch} of 5120 channels x {SCAN.seqlen} steps x {SCAN.dstate} states"},
        "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-channels", type=int, default=64)
    args = ap.parse_args(argv)
    if args.impl == "ours":
        args.warmup = max(args.warmup, 3)   # timing rule: at least 3 untimed warm-up steps
    if args.impl == "reference":
        return bench_reference(args)
    return bench_ours(args)


if __name__ == "__main__":
    main()
