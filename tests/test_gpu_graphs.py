"""The library's calls captured into CUDA graphs and replayed.

A decode loop -- one ssm_state_update (and conv1d_update) per token -- is
launch-bound: each step is a few microseconds of kernel behind host work and
a launch.  Capturing the loop once into a CUDA graph and replaying it removes
that per-step cost.  These tests check that every entry point can be captured
on a torch stream (no host synchronisation, no allocation outside the graph's
pool, cooperative launches and memsets captured as graph nodes) and that a
replay computes exactly what the same calls compute eagerly: bit-for-bit
where the kernels have a fixed summation order, within float32 rounding of
the atomically accumulated gradients.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_util import dev
from selective_state_space_122_b300 import (conv1d_update, device_error, inputs, ssm_scan_bwd, ssm_scan_fwd,
                                            ssm_state_update)

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Warm fn up eagerly (first-call attribute setup), then capture one call
    of it into a graph on a side stream; returns the graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("bt,dim", [(256, 5120), (2, 64)], ids=["bulk-copy", "register"])
def test_decode_chain_graph_equals_eager(bt, dim):
    """64 decode steps captured as one graph (fixed token buffers refilled
    before each replay, the state updated in place) against the same 64
    steps run eagerly from the same state."""
    steps = 64
    d = inputs.make_decode_inputs(inputs.DecodeShape("graph-dec", bt, dim, 16, inputs.BF16), 41)
    toks = [d.token() for _ in range(steps)]
    A, D, bias = dev(d.A), dev(d.D), dev(d.dt_bias)
    tok_dev = [[dev(a) for a in tk] for tk in toks]

    # eager
    st_e = dev(d.state0.copy())
    outs_e = []
    for x, dt, z, B, C in tok_dev:
        outs_e.append(ssm_state_update(st_e, x, dt, A, B, C, D, z, bias, True))
    torch.cuda.synchronize()

    # graph: static buffers for the tokens of every step and for the outputs
    st_g = dev(d.state0.copy())
    stat = [[t.clone() for t in tk] for tk in tok_dev]
    outs_g = [torch.empty_like(tk[0]) for tk in tok_dev]

    def loop():
        for (x, dt, z, B, C), o in zip(stat, outs_g):
            ssm_state_update(st_g, x, dt, A, B, C, D, z, bias, True, out=o)

    st_save = st_g.clone()
    g = _capture(loop)           # the eager warm-up advanced the state (capture does not run)
    st_g.copy_(st_save)
    g.replay()
    torch.cuda.synchronize()
    assert device_error() == 0
    assert torch.equal(st_g, st_e)
    for a, b in zip(outs_g, outs_e):
        assert torch.equal(a, b)
    # a second replay from the same state gives the same result again
    st_g.copy_(st_save)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(st_g, st_e)


def test_conv_and_ssm_decode_step_graph():
    """One token of the SSM half of a Mamba block -- the conv's decode step
    (x -> u with a rolling conv state) then the state update -- captured and
    replayed over 16 tokens by refilling the input buffer."""
    bt, dim, N, W = 64, 1536, 16, 4
    r = np.random.Generator(np.random.PCG64(42))
    d = inputs.make_decode_inputs(inputs.DecodeShape("graph-blk", bt, dim, N, inputs.BF16), 43)
    wconv = dev((r.standard_normal((dim, W)) * 0.5).astype(np.float32))
    bconv = dev((r.standard_normal(dim) * 0.1).astype(np.float32))
    A, D, bias = dev(d.A), dev(d.D), dev(d.dt_bias)
    toks = [[dev(a) for a in d.token()] for _ in range(16)]

    def run(cst, sst, x, dt, z, B, C, u_out=None, y_out=None):
        u = conv1d_update(cst, x, wconv, bconv, True, out=u_out)
        return ssm_state_update(sst, u, dt, A, B, C, D, z, bias, True, out=y_out)

    cst_e = torch.zeros(bt, dim, W - 1, device="cuda")
    sst_e = dev(d.state0.copy())
    ys_e = [run(cst_e, sst_e, *tk) for tk in toks]
    torch.cuda.synchronize()

    cst_g = torch.zeros(bt, dim, W - 1, device="cuda")
    sst_g = dev(d.state0.copy())
    stat = [t.clone() for t in toks[0]]
    u_buf, y_buf = torch.empty_like(stat[0]), torch.empty_like(stat[0])
    saved = (cst_g.clone(), sst_g.clone())
    g = _capture(lambda: run(cst_g, sst_g, *stat, u_out=u_buf, y_out=y_buf))
    cst_g.copy_(saved[0])
    sst_g.copy_(saved[1])
    for tk, y_e in zip(toks, ys_e):
        for dst, src in zip(stat, tk):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y_buf, y_e)
    assert torch.equal(sst_g, sst_e) and torch.equal(cst_g, cst_e)


def test_scan_fwd_and_bwd_graph():
    """The forward scan (tensor-memory path: a cooperative launch after its
    staging kernel) and the backward (three kernels after their memsets),
    each captured once and replayed."""
    shape = inputs.ScanShape("graph-scan", 2, 256, 2048, 16, inputs.BF16)
    inp = inputs.make_scan_inputs(shape, 44)
    r = np.random.Generator(np.random.PCG64(45))
    dout = dev(inputs._activation(r, (shape.batch, shape.seqlen, shape.dim), shape.dtype))
    t = [dev(x) for x in (inp.u, inp.delta, inp.A, inp.B, inp.C, inp.D, inp.z, inp.delta_bias)]

    out_e, last_e = ssm_scan_fwd(*t, True, return_last_state=True)
    out_g, last_g = torch.empty_like(out_e), torch.empty_like(last_e)
    g = _capture(lambda: ssm_scan_fwd(*t, True, out=out_g, last_state=last_g))
    out_g.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert device_error() == 0
    assert torch.equal(out_g, out_e) and torch.equal(last_g, last_e)

    ge = ssm_scan_bwd(*t, True, dout)
    torch.cuda.synchronize()
    res = {}

    def bwd():
        res.update(ssm_scan_bwd(*t, True, dout))

    g2 = _capture(bwd)
    gg = dict(res)               # the graph's output buffers
    for v in gg.values():
        if v is not None:
            v.zero_()
    g2.replay()
    torch.cuda.synchronize()
    assert device_error() == 0
    for k in ("du", "ddelta", "dz"):
        assert torch.equal(gg[k], ge[k]), k           # no atomics: same order
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        torch.testing.assert_close(gg[k], ge[k], rtol=1e-5, atol=1e-6 * float(ge[k].abs().max()))
