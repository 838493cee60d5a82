"""Seeded synthetic inputs for the selective scan and the decode step.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
callers. It draws random numbers and lays them out; it performs none of the
scan's arithmetic.

Recipe (one numpy ``Generator(PCG64(seed))`` per workload):

* draw order: u, delta_raw, z, B, C, dt (-> delta_bias); for the decode
  workload additionally state0, then per-step tokens x, dt, z, B, C;
* every activation is drawn in float32 from N(0, 1) and, for bf16 workloads,
  rounded to bfloat16 with round-to-nearest-even on the host, so the GPU and
  the oracle see bit-identical values;
* A[d, n] = -(n + 1) for every channel (the S4D-real initialisation the Mamba
  block uses; a random negative A is available for robustness cases);
* D = 1 for every channel;
* delta_bias = softplus^-1(dt) with dt log-uniform in [1e-3, 0.1] per
  channel: the "targeted range" initialisation of the Delta projection bias
  named in the state-spaces/mamba docs ("Troubleshoot initialization issues");
* decode state0 ~ N(0, 0.1) (standard deviation 0.1), fp32;
* activations too large to draw on the host (more than 2^31 elements) are
  counter-based instead: uniform on [-1, 1) from an integer hash of the
  element index (below), built on the device in slices and recomputed on the
  host for the channels the oracle checks.

Layouts follow the (batch, length, dim) convention of the Mamba block:
u, delta, z, out are (batch, L, D) channel-contiguous; B and C are
(batch, N, L) time-contiguous, or (batch, G, N, L) with B and C per channel
group (drawn in the same order, G times as many values); A is (D, N); D and
delta_bias are (D,); states are (batch, D, N).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"


@dataclasses.dataclass(frozen=True)
class ScanShape:
    name: str
    batch: int
    dim: int
    seqlen: int
    dstate: int
    dtype: str
    want_last_state: bool = True


# The five workloads: a tiny fp32 case, a Mamba-130M-shaped layer
# (d_model 768, expand 2), a mid-size prefill, a 128K-token long sequence at
# d_model 2560, and a batched decode step.
TINY_F32 = ScanShape("tiny-f32 1x16x64 N4", 1, 16, 64, 4, F32)
LAYER_130M = ScanShape("mamba130m-layer 4x1536x1024 N16", 4, 1536, 1024, 16, BF16)
PREFILL_MID = ScanShape("prefill 8x2048x2048 N16", 8, 2048, 2048, 16, BF16)
LONG_SEQ = ScanShape("long-seq 1x5120x131072 N16", 1, 5120, 131072, 16, BF16)


@dataclasses.dataclass(frozen=True)
class DecodeShape:
    name: str
    batch: int
    dim: int
    dstate: int
    dtype: str


DECODE_256 = DecodeShape("decode 256x5120 N16", 256, 5120, 16, BF16)

SCAN_WORKLOADS = {0: TINY_F32, 1: LAYER_130M, 2: PREFILL_MID, 3: LONG_SEQ}


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even.

    Finite inputs only (the generators never draw NaN); works in 32-bit
    integer arithmetic, in blocks, to keep the temporaries small."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    w_all = x.view(np.uint32).reshape(-1)
    out = np.empty(w_all.shape, np.uint16)
    blk = 1 << 24
    for i in range(0, w_all.size, blk):
        w = w_all[i:i + blk]
        r = (w >> np.uint32(16)) & np.uint32(1)
        r += np.uint32(0x7FFF)
        r += w
        r >>= np.uint32(16)
        out[i:i + blk] = r
    return out.reshape(x.shape)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float64."""
    w = b.astype(np.uint32) << 16
    return w.view(np.float32).astype(np.float64)


def _normal(rng: np.random.Generator, shape, sigma: float = 1.0) -> np.ndarray:
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        out *= np.float32(sigma)
    return out


def _activation(rng, shape, dtype):
    a = _normal(rng, shape)
    return round_to_bf16_bits(a) if dtype == BF16 else a


def _delta_bias(rng, dim, dt_min=1e-3, dt_max=0.1):
    lo, hi = np.log(dt_min), np.log(dt_max)
    dt = np.exp(rng.uniform(lo, hi, size=dim))            # float64
    # softplus^-1(dt) = log(exp(dt) - 1) = dt + log(-expm1(-dt)), in float64
    inv = dt + np.log(-np.expm1(-dt))
    return inv.astype(np.float32)


def a_s4d_real(dim: int, dstate: int) -> np.ndarray:
    """A[d, n] = -(n + 1), float32, shape (dim, dstate)."""
    return np.tile(-np.arange(1, dstate + 1, dtype=np.float32), (dim, 1))


def a_random(rng: np.random.Generator, dim: int, dstate: int) -> np.ndarray:
    """A = -exp(N(0, 1)): unstructured negative real A (robustness cases)."""
    return (-np.exp(rng.standard_normal((dim, dstate)))).astype(np.float32)


@dataclasses.dataclass
class ScanInputs:
    shape: ScanShape
    u: np.ndarray          # (batch, L, D)   f32 or bf16 bits (uint16)
    delta: np.ndarray      # (batch, L, D)
    z: Optional[np.ndarray]
    B: np.ndarray          # (batch, N, L), or (batch, G, N, L) per channel group
    C: np.ndarray          # same shape as B
    A: np.ndarray          # (D, N) f32
    D: Optional[np.ndarray]
    delta_bias: Optional[np.ndarray]
    softplus: bool = True

    def channels(self, sel) -> "ScanInputs":
        """The same inputs restricted to the channels ``sel`` (no arithmetic)."""
        sel = np.asarray(sel)
        pick = lambda a: None if a is None else np.ascontiguousarray(a[:, :, sel])
        vec = lambda a: None if a is None else np.ascontiguousarray(a[sel])
        shape = dataclasses.replace(self.shape, dim=int(sel.size))
        return ScanInputs(shape, pick(self.u), pick(self.delta), pick(self.z), self.B, self.C,
                          vec(self.A), vec(self.D), vec(self.delta_bias), self.softplus)

    def as_f64(self) -> dict:
        """Exact float64 copies of every input (for the oracle)."""
        w = bf16_bits_to_f64 if self.shape.dtype == BF16 else (lambda a: a.astype(np.float64))
        f = lambda a: None if a is None else a.astype(np.float64)
        return dict(u=w(self.u), delta=w(self.delta), z=None if self.z is None else w(self.z),
                    B=w(self.B), C=w(self.C), A=f(self.A), D=f(self.D),
                    delta_bias=f(self.delta_bias), softplus=self.softplus)


def make_scan_inputs(shape: ScanShape, seed: int, *, random_a: bool = False,
                     with_z: bool = True, with_d: bool = True,
                     with_bias: bool = True, softplus: bool = True, ngroups: int = 1) -> ScanInputs:
    """Seeded inputs for a full-sequence scan of ``shape``; ngroups > 1 draws
    B and C per channel group, shaped (batch, ngroups, N, L)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    bt, L, D, N, dt = shape.batch, shape.seqlen, shape.dim, shape.dstate, shape.dtype
    u = _activation(rng, (bt, L, D), dt)
    delta = _activation(rng, (bt, L, D), dt)
    z = _activation(rng, (bt, L, D), dt)
    bc = (bt, N, L) if ngroups == 1 else (bt, ngroups, N, L)
    B = _activation(rng, bc, dt)
    C = _activation(rng, bc, dt)
    bias = _delta_bias(rng, D)
    A = a_random(rng, D, N) if random_a else a_s4d_real(D, N)
    return ScanInputs(shape, u, delta, z if with_z else None, B, C, A,
                      np.ones(D, np.float32) if with_d else None,
                      bias if with_bias else None, softplus)


@dataclasses.dataclass
class DecodeInputs:
    shape: DecodeShape
    state0: np.ndarray     # (batch, D, N) f32
    A: np.ndarray
    D: np.ndarray
    dt_bias: np.ndarray
    rng: np.random.Generator

    def token(self, ngroups: int = 1):
        """Next token: x, dt, z (batch, D) and B, C (batch, N), or (batch,
        ngroups, N) per channel group, in the workload dtype."""
        s = self.shape
        x = _activation(self.rng, (s.batch, s.dim), s.dtype)
        dt = _activation(self.rng, (s.batch, s.dim), s.dtype)
        z = _activation(self.rng, (s.batch, s.dim), s.dtype)
        bc = (s.batch, s.dstate) if ngroups == 1 else (s.batch, ngroups, s.dstate)
        B = _activation(self.rng, bc, s.dtype)
        C = _activation(self.rng, bc, s.dtype)
        return x, dt, z, B, C


def make_decode_inputs(shape: DecodeShape, seed: int) -> DecodeInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    bias = _delta_bias(rng, shape.dim)
    state0 = _normal(rng, (shape.batch, shape.dim, shape.dstate), sigma=0.1)
    return DecodeInputs(shape, state0, a_s4d_real(shape.dim, shape.dstate),
                        np.ones(shape.dim, np.float32), bias, rng)


# ------------------------------------------------------------------
# Counter-based draws, for activations too large to draw on the host.
#
# Value i of stream s under seed k is a pure function of (k, s, i): the
# 64-bit element index i (row-major over (batch, L, D)) is hashed with
# C. Wellons' "lowbias32" integer hash ("Prospecting for Hash Functions",
# 2018), and the top 24 bits of the hash give a uniform value on [-1, 1)
# with 2^-23 spacing, exact in float32.  The same code runs on numpy int64
# arrays (the oracle's sampled channels) and on torch int64 tensors (the
# full tensors, built on the device in slices), and gives bit-identical
# values on both: every step is an integer operation whose intermediate
# results stay below 2^49, then one exact conversion and scaling in float32.

_M32 = 0xFFFFFFFF


def _mul32(x, c: int):
    """(x * c) mod 2^32 for integers 0 <= x < 2^32, with c split in 16-bit
    halves so that no product exceeds 2^49 (no signed 64-bit overflow)."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def _lowbias32(x):
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    return x ^ (x >> 16)


def counter_bits(index, stream: int, seed: int):
    """32-bit hash of (seed, stream, index) for a non-negative int64 index
    array or tensor (either library)."""
    key = int(_lowbias32(((seed & _M32) * 0x9E3779B9 + stream) & _M32))
    return _lowbias32((index & _M32) ^ _lowbias32((index >> 32) ^ key))


def counter_uniform_np(index: np.ndarray, stream: int, seed: int) -> np.ndarray:
    """Uniform [-1, 1) float32 values for an int64 index array."""
    h = counter_bits(np.asarray(index, dtype=np.int64), stream, seed)
    return (h >> 8).astype(np.float32) * np.float32(2.0 ** -23) - np.float32(1.0)


def counter_uniform_torch(index, stream: int, seed: int):
    """The same values for an int64 torch tensor (on any device)."""
    import torch
    h = counter_bits(index, stream, seed)
    return (h >> 8).to(torch.float32) * (2.0 ** -23) - 1.0


def counter_activation_channels(batch: int, seqlen: int, dim: int, sel, stream: int, seed: int,
                                dtype: str) -> np.ndarray:
    """Channels ``sel`` of the (batch, seqlen, dim) counter-drawn activation
    (bf16 bits or float32), shaped (batch, seqlen, len(sel))."""
    sel = np.asarray(sel, dtype=np.int64)
    rows = np.arange(batch * seqlen, dtype=np.int64).reshape(batch, seqlen, 1)
    v = counter_uniform_np(rows * dim + sel.reshape(1, 1, -1), stream, seed)
    return round_to_bf16_bits(v) if dtype == BF16 else v


def counter_activation_device(batch: int, seqlen: int, dim: int, stream: int, seed: int, dtype: str,
                              device, rows_per_slice: int = 8192):
    """The whole (batch, seqlen, dim) counter-drawn activation as a torch
    tensor on ``device`` (bfloat16 or float32), built slice by slice."""
    import torch
    tdt = torch.bfloat16 if dtype == BF16 else torch.float32
    out = torch.empty((batch, seqlen, dim), dtype=tdt, device=device)
    col = torch.arange(dim, dtype=torch.int64, device=device).reshape(1, -1)
    for b in range(batch):
        for t0 in range(0, seqlen, rows_per_slice):
            t1 = min(seqlen, t0 + rows_per_slice)
            rows = torch.arange(b * seqlen + t0, b * seqlen + t1, dtype=torch.int64, device=device).reshape(-1, 1)
            out[b, t0:t1] = counter_uniform_torch(rows * dim + col, stream, seed).to(tdt)
    return out
