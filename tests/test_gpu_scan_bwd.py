"""The scan's backward (ssm_scan_bwd) against the float64 adjoint oracle."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev, host_f64
from selective_state_space_122_b300 import inputs, ssm_scan_bwd, ssm_scan_fwd

pytestmark = pytest.mark.gpu


def _close(got, ref, rel, what, rounded=False):
    """|got - ref| <= rel * max(rms(ref), max|ref| / 50) elementwise (gradients
    that sum many terms are compared on the scale of the whole tensor), plus
    the half-ulp 2^-8 |ref| of a bf16 output when ``rounded``."""
    got = np.asarray(got, dtype=np.float64)
    scale = max(float(np.sqrt(np.mean(ref ** 2))), float(np.max(np.abs(ref))) / 50.0, 1e-30)
    bound = rel * scale + (2.0 ** -8 * np.abs(ref) if rounded else 0.0)
    excess = np.abs(got - ref) - bound
    assert float(np.max(excess)) <= 0.0, (f"{what}: max|err| {float(np.max(np.abs(got - ref))):.3e}, "
                                          f"bound {rel:.0e} x {scale:.3e}")


@pytest.mark.parametrize("bt,dim,L,N,dtype,kw", [
    (2, 24, 77, 16, inputs.F32, {}),
    (1, 40, 100, 8, inputs.F32, dict(softplus=False)),
    (2, 70, 65, 4, inputs.F32, dict(with_z=False, with_d=False, with_bias=False)),
    (2, 64, 300, 16, inputs.BF16, {}),
    (3, 48, 129, 8, inputs.BF16, dict(random_a=True)),
    (1, 16, 1, 16, inputs.F32, {}),
    (2, 256, 2048, 16, inputs.BF16, {}),
    # several segments per chain (the aggregates carry the state and the
    # adjoint across them), ragged last segment and chunk, ragged channels
    (2, 64, 1000, 16, inputs.BF16, {}),
    (1, 96, 777, 8, inputs.F32, {}),
    (2, 130, 600, 4, inputs.BF16, dict(random_a=True)),
    # odd channel count: element-wise staging and stores
    (1, 37, 1100, 16, inputs.BF16, {}),
    (1, 45, 530, 16, inputs.F32, dict(with_z=False)),
])
def test_scan_bwd_matches_adjoint_oracle(bt, dim, L, N, dtype, kw):
    inp = inputs.make_scan_inputs(inputs.ScanShape("bwd", bt, dim, L, N, dtype), 1200 + dim + L, **kw)
    if not inp.softplus:
        # without softplus the raw timestep is used as is: keep it positive and
        # small so the recurrence stays bounded (float32 cases only)
        assert dtype == inputs.F32
        inp = dataclasses.replace(inp, delta=(np.abs(inp.delta) * 0.05).astype(np.float32), delta_bias=None)
    r = np.random.Generator(np.random.PCG64(1300 + L))
    dout = inputs._activation(r, (bt, L, dim), dtype)
    f = inp.as_f64()
    dout_f = inputs.bf16_bits_to_f64(dout) if dtype == inputs.BF16 else dout.astype(np.float64)
    ref = oracle.scan_bwd(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"], f["delta_bias"],
                          f["softplus"], dout_f)
    g = ssm_scan_bwd(dev(inp.u), dev(inp.delta), dev(inp.A), dev(inp.B), dev(inp.C), dev(inp.D), dev(inp.z),
                     dev(inp.delta_bias), inp.softplus, dev(dout))
    torch.cuda.synchronize()
    # float32 math throughout; bf16 outputs (du, ddelta, dz) carry their own rounding
    bf = dtype == inputs.BF16
    for k in ("du", "ddelta", "dz"):
        if ref[k] is not None:
            _close(host_f64(g[k]), ref[k], 1e-4, k, rounded=bf)
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        if ref[k] is not None:
            _close(host_f64(g[k]), ref[k], 1e-4, k)


def test_scan_bwd_prefill_shape():
    """The mid-size prefill shape (8 x 2048 x 2048, d_state 16, bf16) in one
    call -- 512 CTAs under the 4-CTA register budget -- against the adjoint
    oracle on every output element."""
    bt, dim, L, N, dtype = 8, 2048, 2048, 16, inputs.BF16
    inp = inputs.make_scan_inputs(inputs.PREFILL_MID, 1400)
    r = np.random.Generator(np.random.PCG64(1401))
    dout = inputs._activation(r, (bt, L, dim), dtype)
    g = ssm_scan_bwd(dev(inp.u), dev(inp.delta), dev(inp.A), dev(inp.B), dev(inp.C), dev(inp.D), dev(inp.z),
                     dev(inp.delta_bias), inp.softplus, dev(dout))
    torch.cuda.synchronize()
    f = inp.as_f64()
    ref = oracle.scan_bwd(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"], f["delta_bias"],
                          f["softplus"], inputs.bf16_bits_to_f64(dout))
    for k in ("du", "ddelta", "dz"):
        _close(host_f64(g[k]), ref[k], 1e-4, k, rounded=True)
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        _close(host_f64(g[k]), ref[k], 1e-4, k)


@pytest.mark.parametrize("bt,dim,L,N,dtype,G,given", [
    (2, 64, 300, 16, inputs.BF16, 1, "both"),
    (1, 40, 100, 8, inputs.F32, 2, "both"),
    (2, 96, 129, 4, inputs.F32, 1, "both"),
    (2, 128, 77, 16, inputs.BF16, 4, "both"),
    # several segments per chain
    (2, 64, 1001, 16, inputs.BF16, 2, "both"),
    # one of the two alone (the other is zero), dL/d initial_state requested,
    # L not a multiple of the 8-step chunk
    (2, 64, 301, 16, inputs.BF16, 1, "initial_state"),
    (1, 48, 900, 8, inputs.F32, 2, "initial_state"),
    (2, 64, 301, 16, inputs.BF16, 1, "dlast"),
    (1, 48, 899, 8, inputs.F32, 2, "dlast"),
])
def test_scan_bwd_from_state(bt, dim, L, N, dtype, G, given):
    """The backward of the scan from a given state whose final state enters the
    loss (ssm_scan_bwd_from_state) against the oracle, dL/d initial_state
    included; with only one of initial_state and dlast given, the oracle takes
    the missing one as zero."""
    inp = inputs.make_scan_inputs(inputs.ScanShape("bwd-h0", bt, dim, L, N, dtype), 1500 + dim + L, ngroups=G)
    r = np.random.Generator(np.random.PCG64(1600 + L))
    dout = inputs._activation(r, (bt, L, dim), dtype)
    h0 = (r.standard_normal((bt, dim, N)) * 0.5).astype(np.float32)
    dlast = r.standard_normal((bt, dim, N)).astype(np.float32)
    if given == "initial_state":
        dlast = None
    elif given == "dlast":
        h0 = None
    f = inp.as_f64()
    dout_f = inputs.bf16_bits_to_f64(dout) if dtype == inputs.BF16 else dout.astype(np.float64)
    zero = np.zeros((bt, dim, N))
    ref = oracle.scan_bwd(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"], f["delta_bias"],
                          f["softplus"], dout_f, initial_state=zero if h0 is None else h0.astype(np.float64),
                          dlast=zero if dlast is None else dlast.astype(np.float64))
    g = ssm_scan_bwd(dev(inp.u), dev(inp.delta), dev(inp.A), dev(inp.B), dev(inp.C), dev(inp.D), dev(inp.z),
                     dev(inp.delta_bias), inp.softplus, dev(dout),
                     initial_state=None if h0 is None else dev(h0), dlast=None if dlast is None else dev(dlast))
    torch.cuda.synchronize()
    bf = dtype == inputs.BF16
    for k in ("du", "ddelta", "dz"):
        _close(host_f64(g[k]), ref[k], 1e-4, k, rounded=bf)
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias", "dinitial_state"):
        _close(host_f64(g[k]), ref[k], 1e-4, k)


def test_scan_bwd_long_sequence_sampled_channels():
    """The backward at the long-sequence size (1 x 5120 x 131072, d_state 16,
    bf16): the chains cut into the maximum of 64 segments of 256 chunks.
    Every per-channel gradient of 16 sampled channels -- du, ddelta, dz over
    all 128K steps, dA, dD, ddelta_bias -- against the adjoint oracle run on
    those channels alone.  dB and dC sum over every channel, so they are held
    to the identity <dB, B> = <dC, C> = sum(dout * (out - D u silu(z))) (out
    is linear in B and in C apart from the D u term), with out from the
    forward scan and a bound on its bf16 rounding."""
    shape = inputs.LONG_SEQ
    inp = inputs.make_scan_inputs(shape, 31)
    r = np.random.Generator(np.random.PCG64(32))
    dout = inputs._activation(r, (shape.batch, shape.seqlen, shape.dim), shape.dtype)
    t = dict(u=dev(inp.u), delta=dev(inp.delta), A=dev(inp.A), B=dev(inp.B), C=dev(inp.C), D=dev(inp.D),
             z=dev(inp.z), bias=dev(inp.delta_bias))
    do = dev(dout)
    g = ssm_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["bias"], inp.softplus, do)
    torch.cuda.synchronize()
    sel = np.array([0, 1, 31, 32, 33, 127, 128, 1000, 2047, 2560, 3333, 4095, 4096, 5087, 5118, 5119])
    f = inp.channels(sel).as_f64()
    dsel = inputs.bf16_bits_to_f64(np.ascontiguousarray(dout[:, :, sel]))
    ref = oracle.scan_bwd(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"], f["delta_bias"],
                          f["softplus"], dsel)
    idx = torch.as_tensor(sel, device=do.device)
    for k in ("du", "ddelta", "dz"):
        _close(host_f64(g[k][:, :, idx]), ref[k], 1e-4, k, rounded=True)
    _close(host_f64(g["dA"][idx]), ref["dA"], 1e-4, "dA")
    for k in ("dD", "ddelta_bias"):
        _close(host_f64(g[k][idx]), ref[k], 1e-4, k)
    for k in ("dB", "dC"):
        assert bool(torch.isfinite(g[k]).all()), k
    # the B/C identity against the forward scan's output
    del g["du"], g["ddelta"], g["dz"]
    out, _ = ssm_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["bias"], inp.softplus)
    torch.cuda.synchronize()
    dof = do.double()
    uu, zz = t["u"].double(), t["z"].double()
    skip = t["D"].double() * uu * zz * torch.sigmoid(zz)
    terms = dof * out.double()
    rhs = float((terms - dof * skip).sum())
    lhs_b = float((g["dB"].double() * t["B"].double()).sum())
    lhs_c = float((g["dC"].double() * t["C"].double()).sum())
    # out is rounded to bf16 (error <= 2^-8 |out|, roughly uniform): six
    # standard deviations of the rounding's contribution to the sum
    bound = 6.0 * 2.0 ** -8 / np.sqrt(3.0) * float(torch.sqrt((terms ** 2).sum())) + 1e-4 * abs(rhs)
    assert abs(lhs_b - rhs) <= bound, (lhs_b, rhs, bound)
    assert abs(lhs_c - rhs) <= bound, (lhs_c, rhs, bound)
