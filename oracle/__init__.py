"""ctypes front end of the float64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline / reference leg use this package to check and to time the CUDA
library.  The library never imports it, and it imports nothing from the
library.  ``build()`` compiles ``oracle.c`` with gcc (plain -O2, no fast-math,
no FP contraction, OpenMP only across independent channels).

Every function here takes and returns float64 numpy arrays in the layouts that
``oracle.c`` documents; callers widen bf16/fp32 inputs exactly before calling.
Every oracle function is pinned by ``tests/test_oracle_pins.py`` (brute-force
sums, the time-invariant convolution closed form, a log-depth associative
scan, limiting cases and invariances); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.c")
LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math"]

_lib = None


def build(src: str = SRC, out: str = LIB, extra: Optional[list] = None) -> str:
    """Compile the oracle into a shared library and return its path."""
    cmd = ["gcc", *CFLAGS, *(extra or []), "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def load(path: Optional[str] = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    p = path or LIB
    if path is None and (not os.path.exists(p) or os.path.getmtime(p) < os.path.getmtime(SRC)):
        build()
    lib = ctypes.CDLL(p)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_scan.argtypes = [dp] * 8 + [ctypes.c_int, dp, dp] + [ctypes.c_int] * 4
    lib.oracle_scan.restype = ctypes.c_int
    lib.oracle_scan_from.argtypes = [dp] * 8 + [ctypes.c_int, dp, dp, dp] + [ctypes.c_int] * 4
    lib.oracle_scan_from.restype = ctypes.c_int
    lib.oracle_scan_bwd.argtypes = [dp] * 8 + [ctypes.c_int] + [dp] * 9 + [ctypes.c_int] * 4
    lib.oracle_scan_bwd.restype = ctypes.c_int
    lib.oracle_conv1d.argtypes = [dp, dp, dp, ctypes.c_int, dp, dp, dp] + [ctypes.c_int] * 4
    lib.oracle_conv1d.restype = ctypes.c_int
    lib.oracle_conv1d_update.argtypes = [dp, dp, dp, dp, ctypes.c_int, dp] + [ctypes.c_int] * 3
    lib.oracle_conv1d_update.restype = ctypes.c_int
    lib.oracle_step.argtypes = [dp] * 9 + [ctypes.c_int, dp] + [ctypes.c_int] * 3
    lib.oracle_step.restype = ctypes.c_int
    lib.oracle_scan_grouped.argtypes = [dp] * 8 + [ctypes.c_int, dp, dp, dp] + [ctypes.c_int] * 5
    lib.oracle_scan_grouped.restype = ctypes.c_int
    lib.oracle_step_grouped.argtypes = [dp] * 9 + [ctypes.c_int, dp] + [ctypes.c_int] * 4
    lib.oracle_step_grouped.restype = ctypes.c_int
    lib.oracle_scan_bwd_grouped.argtypes = [dp] * 8 + [ctypes.c_int] + [dp] * 9 + [ctypes.c_int] * 5
    lib.oracle_scan_bwd_grouped.restype = ctypes.c_int
    lib.oracle_scan_bwd_from.argtypes = ([dp] * 8 + [ctypes.c_int] + [dp] * 3 + [dp] * 9
                                         + [ctypes.c_int] * 5)
    lib.oracle_scan_bwd_from.restype = ctypes.c_int
    lib.oracle_softplus.argtypes = [ctypes.c_double]
    lib.oracle_softplus.restype = ctypes.c_double
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _p(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"], "oracle takes C-contiguous float64"
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _groups(B, lead, tail):
    """Number of B/C groups: B is lead + (N, ...) for one group, lead +
    (ngroups, N, ...) for several."""
    return 1 if B.ndim == len(lead) + 1 + len(tail) else B.shape[len(lead)]


def scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
         want_last_state=True, lib=None, initial_state=None):
    """Full-sequence selective scan.

    u, delta, z: (batch, L, dim); B, C: (batch, N, L), or (batch, ngroups, N, L)
    with channel d reading group d // (dim // ngroups); A: (dim, N);
    D, delta_bias: (dim,); initial_state: (batch, dim, N) or None (zero).
    Returns (out (batch, L, dim), last_state (batch, dim, N) or None), float64.
    """
    lib = lib or load()
    u, delta, A, B, C, D, z, delta_bias, h0 = map(_f64, (u, delta, A, B, C, D, z, delta_bias, initial_state))
    bt, L, dim = u.shape
    N = A.shape[1]
    G = _groups(B, (bt,), (L,))
    assert delta.shape == u.shape and A.shape == (dim, N)
    shape = (bt, N, L) if B.ndim == 3 else (bt, G, N, L)
    assert B.shape == shape and C.shape == shape
    assert h0 is None or h0.shape == (bt, dim, N)
    out = np.empty_like(u)
    last = np.empty((bt, dim, N)) if want_last_state else None
    rc = lib.oracle_scan_grouped(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
                                 int(bool(softplus)), _p(h0), _p(out), _p(last), bt, dim, L, N, G)
    if rc != 0:
        raise ValueError(f"oracle_scan rejected its arguments (code {rc})")
    return out, last


def step(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=True, lib=None):
    """One recurrent update.  ``state`` (batch, dim, N) float64 is updated in
    place; x, dt, z: (batch, dim); B, C: (batch, N) or (batch, ngroups, N).
    Returns out (batch, dim)."""
    lib = lib or load()
    assert state.dtype == np.float64 and state.flags["C_CONTIGUOUS"]
    x, dt, A, B, C, D, z, dt_bias = map(_f64, (x, dt, A, B, C, D, z, dt_bias))
    bt, dim, N = state.shape
    G = _groups(B, (bt,), ())
    assert B.shape == C.shape and B.shape[-1] == N
    out = np.empty((bt, dim))
    rc = lib.oracle_step_grouped(_p(state), _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(z),
                                 _p(dt_bias), int(bool(dt_softplus)), _p(out), bt, dim, N, G)
    if rc != 0:
        raise ValueError(f"oracle_step rejected its arguments (code {rc})")
    return out


def scan_bwd(u, delta, A, B, C, D, z, delta_bias, softplus, dout, lib=None, initial_state=None, dlast=None):
    """Gradients of L = sum(dout * out) of the scan (from h = 0) with respect to
    every input.  Returns a dict du, ddelta (batch, L, dim); dA (dim, N); dB, dC
    shaped like B and C ((batch, N, L) or (batch, ngroups, N, L)); dD,
    ddelta_bias (dim,) or None; dz (batch, L, dim) or None.

    initial_state (batch, dim, N) starts the forward scan from that state, and
    dlast (batch, dim, N) is dL/d last_state (the final state's part of the
    loss); both default to zero.  The dict also holds dinitial_state =
    dL/d initial_state (batch, dim, N)."""
    lib = lib or load()
    u, delta, A, B, C, D, z, delta_bias, dout = map(_f64, (u, delta, A, B, C, D, z, delta_bias, dout))
    h0, dl = _f64(initial_state), _f64(dlast)
    bt, L, dim = u.shape
    N = A.shape[1]
    G = _groups(B, (bt,), (L,))
    assert B.shape == C.shape and B.shape[-2:] == (N, L)
    g = dict(du=np.empty_like(u), ddelta=np.empty_like(u), dA=np.empty_like(A), dB=np.empty_like(B),
             dC=np.empty_like(C), dD=None if D is None else np.empty(dim),
             dz=None if z is None else np.empty_like(u),
             ddelta_bias=None if delta_bias is None else np.empty(dim), dinitial_state=np.empty((bt, dim, N)))
    for a in (h0, dl):
        assert a is None or a.shape == (bt, dim, N)
    rc = lib.oracle_scan_bwd_from(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
                                  int(bool(softplus)), _p(h0), _p(dout), _p(dl), _p(g["du"]), _p(g["ddelta"]),
                                  _p(g["dA"]), _p(g["dB"]), _p(g["dC"]), _p(g["dD"]), _p(g["dz"]),
                                  _p(g["ddelta_bias"]), _p(g["dinitial_state"]), bt, dim, L, N, G)
    if rc != 0:
        raise ValueError(f"oracle_scan_bwd rejected its arguments (code {rc})")
    return g


def conv1d(x, w, bias=None, silu=True, state_in=None, want_state=True, lib=None):
    """Depthwise causal convolution (+ SiLU).  x: (batch, L, dim); w: (dim, W);
    bias: (dim,); state_in: (batch, dim, W-1) or None (zeros).  Returns
    (out (batch, L, dim), state_out (batch, dim, W-1) or None), float64."""
    lib = lib or load()
    x, w, bias, state_in = map(_f64, (x, w, bias, state_in))
    bt, L, dim = x.shape
    W = w.shape[1]
    assert w.shape == (dim, W) and (state_in is None or state_in.shape == (bt, dim, W - 1))
    out = np.empty_like(x)
    st = np.empty((bt, dim, W - 1)) if want_state else None
    rc = lib.oracle_conv1d(_p(x), _p(w), _p(bias), int(bool(silu)), _p(state_in), _p(out), _p(st),
                           bt, dim, L, W)
    if rc != 0:
        raise ValueError(f"oracle_conv1d rejected its arguments (code {rc})")
    return out, st


def conv1d_update(state, x, w, bias=None, silu=True, lib=None):
    """One decode step; ``state`` (batch, dim, W-1) float64 is updated in place.
    x: (batch, dim).  Returns out (batch, dim)."""
    lib = lib or load()
    assert state.dtype == np.float64 and state.flags["C_CONTIGUOUS"]
    x, w, bias = map(_f64, (x, w, bias))
    bt, dim = x.shape
    W = w.shape[1]
    out = np.empty_like(x)
    rc = lib.oracle_conv1d_update(_p(state), _p(x), _p(w), _p(bias), int(bool(silu)), _p(out), bt, dim, W)
    if rc != 0:
        raise ValueError(f"oracle_conv1d_update rejected its arguments (code {rc})")
    return out


def softplus(x: float, lib=None) -> float:
    return (lib or load()).oracle_softplus(float(x))


def silu(x: float, lib=None) -> float:
    return (lib or load()).oracle_silu(float(x))


def set_threads(n: int, lib=None) -> None:
    (lib or load()).oracle_set_threads(int(n))


def max_threads(lib=None) -> int:
    return (lib or load()).oracle_max_threads()
