"""B and C per channel group (ssm_scan_fwd_grouped, ssm_state_update_grouped,
ssm_scan_bwd_grouped) against the float64 oracle, on every kernel path that
takes the group size, plus the identity "identical groups = one group"."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_out, check_state, dev, host_f64, paths, scan_layout
from selective_state_space_122_b300 import SSMError, device_error, inputs, ssm_scan_bwd, ssm_scan_fwd
from selective_state_space_122_b300 import ssm_state_update
from test_gpu_scan_bwd import _close as grad_close

pytestmark = pytest.mark.gpu


def grouped_paths(N, dim, gch, dtype):
    """The paths that take groups of gch channels: the tensor-memory kernels
    need whole 32-channel blocks in a group, the segmented kernel whole
    blocks of 128 / N channels; the generic layouts take any size."""
    out = []
    for g in paths(N, dim, dtype):
        if g in ("ws", "tmem2") and gch % 32:
            continue
        if g == "seg" and gch % (128 // N):
            continue
        out.append(g)
    return out


def _device(inp):
    return {k: dev(getattr(inp, k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias")}


def _scan(t, softplus, initial_state=None):
    out, last = ssm_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                             softplus, return_last_state=True, initial_state=initial_state)
    torch.cuda.synchronize()
    assert device_error() == 0, "a scan kernel reported a timed-out wait"
    return out, last


def _oracle(inp, h0=None):
    f = inp.as_f64()
    return oracle.scan(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"], f["delta_bias"],
                       f["softplus"], initial_state=h0)


@pytest.mark.parametrize("bt,dim,L,N,dtype,G", [
    (2, 128, 300, 16, inputs.BF16, 4),     # 32 channels per group: every path
    (2, 256, 200, 16, inputs.BF16, 2),
    (2, 72, 130, 16, inputs.BF16, 9),      # 8 per group: segmented, generic
    (2, 30, 77, 16, inputs.BF16, 10),      # 3 per group (odd): generic only
    (3, 64, 65, 8, inputs.F32, 4),         # 16 per group
    (2, 64, 50, 4, inputs.F32, 2),         # 32 per group
    (1, 96, 100, 8, inputs.BF16, 12),      # 8 per group, below the 8-state block of 16
    (2, 40, 33, 4, inputs.F32, 40),        # one channel per group
])
def test_grouped_scan_every_path(bt, dim, L, N, dtype, G):
    inp = inputs.make_scan_inputs(inputs.ScanShape("grp", bt, dim, L, N, dtype), 2000 + dim + L, ngroups=G)
    assert inp.B.shape == (bt, G, N, L)
    ref, ref_last = _oracle(inp)
    t = _device(inp)
    gp = grouped_paths(N, dim, dim // G, dtype)
    for g in [None] + gp:
        with scan_layout(g):
            out, last = _scan(t, inp.softplus)
        check_out(host_f64(out), ref, dtype, f"grouped out, path {g}")
        check_state(host_f64(last), ref_last, dtype, f"grouped state, path {g}")


@pytest.mark.parametrize("path", ["tmem2", "ws", "seg"])
def test_fast_path_rejects_group_sizes_it_cannot_take(path):
    """Forcing a kernel onto groups that split its channel block is
    SSM_ERR_UNSUPPORTED, before anything is launched."""
    inp = inputs.make_scan_inputs(inputs.ScanShape("grp-rej", 2, 64, 64, 16, inputs.BF16), 2100, ngroups=16)
    t = _device(inp)                       # 4 channels per group
    with scan_layout(path), pytest.raises(SSMError) as e:
        _scan(t, inp.softplus)
    assert e.value.code == 4


@pytest.mark.parametrize("path", [None, "tmem2", "ws", "seg"])
def test_grouped_long_multisegment(path):
    """Many segments per chain with 8 groups of 640 channels, checked on
    sampled channels of every group against the oracle of that group."""
    bt, dim, L, N, G = 1, 5120, 4096, 16, 8
    inp = inputs.make_scan_inputs(inputs.ScanShape("grp-long", bt, dim, L, N, inputs.BF16), 2200, ngroups=G)
    h0 = (np.random.Generator(np.random.PCG64(2201)).standard_normal((bt, dim, N)) * 0.5).astype(np.float32)
    t = _device(inp)
    with scan_layout(path):
        out, last = _scan(t, inp.softplus, torch.from_numpy(h0).cuda())
    gch = dim // G
    for g in range(G):
        sel = np.arange(g * gch + (g % 5), (g + 1) * gch, 61)
        sub = dataclasses.replace(inp.channels(sel), B=np.ascontiguousarray(inp.B[:, g]),
                                  C=np.ascontiguousarray(inp.C[:, g]))
        ref, ref_last = _oracle(sub, h0[:, sel].astype(np.float64))
        idx = torch.as_tensor(sel, device=out.device)
        check_out(host_f64(out[:, :, idx]), ref, inputs.BF16, f"group {g} out, path {path}")
        check_state(host_f64(last[:, idx]), ref_last, inputs.BF16, f"group {g} state, path {path}")


@pytest.mark.parametrize("path", [None, "seg", 2])
def test_identical_groups_equal_one_group(path):
    """B and C repeated over 4 groups give exactly the one-group result: every
    channel sees the same values in the same order of operations."""
    inp = inputs.make_scan_inputs(inputs.ScanShape("grp-same", 2, 256, 500, 16, inputs.BF16), 2300)
    t = _device(inp)
    with scan_layout(path):
        o1, s1 = _scan(t, inp.softplus)
        t4 = dict(t, B=t["B"][:, None].repeat(1, 4, 1, 1).contiguous(), C=t["C"][:, None].repeat(1, 4, 1, 1).contiguous())
        o4, s4 = _scan(t4, inp.softplus)
    assert torch.equal(o1, o4) and torch.equal(s1, s4)


def f64(a, dtype):
    return inputs.bf16_bits_to_f64(a) if dtype == inputs.BF16 else a.astype(np.float64)


@pytest.mark.parametrize("dtype,N,bt,dim,G", [(inputs.BF16, 16, 64, 5120, 8), (inputs.F32, 8, 3, 48, 3),
                                               (inputs.BF16, 4, 5, 30, 10), (inputs.F32, 16, 2, 7, 7),
                                               # bulk-copy pipeline, groups crossing its tiles
                                               (inputs.BF16, 16, 160, 200, 4), (inputs.F32, 8, 200, 192, 6)])
def test_grouped_decode_step(dtype, N, bt, dim, G):
    d = inputs.make_decode_inputs(inputs.DecodeShape("grp-step", bt, dim, N, dtype), 2400 + dim)
    x, dt, z, B, C = d.token(ngroups=G)
    assert B.shape == (bt, G, N)
    state = dev(d.state0.copy())
    out = ssm_state_update(state, dev(x), dev(dt), dev(d.A), dev(B), dev(C), dev(d.D), dev(z), dev(d.dt_bias), True)
    torch.cuda.synchronize()
    ref_state = d.state0.astype(np.float64)
    ref = oracle.step(ref_state, f64(x, dtype), f64(dt, dtype), d.A, f64(B, dtype), f64(C, dtype), d.D,
                      f64(z, dtype), d.dt_bias, True)
    check_out(host_f64(out), ref, dtype)
    check_state(host_f64(state), ref_state, dtype, "grouped decode state")


@pytest.mark.parametrize("bt,dim,L,N,dtype,G", [
    (2, 64, 300, 16, inputs.BF16, 4),
    (2, 48, 77, 8, inputs.F32, 3),
    (1, 30, 65, 16, inputs.F32, 10),       # 3 channels per group
    (2, 256, 1024, 16, inputs.BF16, 2),
    # several segments per chain, groups narrower than the 64- and 128-channel
    # blocks of d_state 8 and 4
    (1, 96, 2000, 8, inputs.BF16, 3),
    (1, 200, 1500, 4, inputs.F32, 5),
])
def test_grouped_bwd(bt, dim, L, N, dtype, G):
    inp = inputs.make_scan_inputs(inputs.ScanShape("grp-bwd", bt, dim, L, N, dtype), 2500 + dim + L, ngroups=G)
    r = np.random.Generator(np.random.PCG64(2600 + L))
    dout = inputs._activation(r, (bt, L, dim), dtype)
    f = inp.as_f64()
    ref = oracle.scan_bwd(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"], f["delta_bias"],
                          f["softplus"], f64(dout, dtype))
    g = ssm_scan_bwd(dev(inp.u), dev(inp.delta), dev(inp.A), dev(inp.B), dev(inp.C), dev(inp.D), dev(inp.z),
                     dev(inp.delta_bias), inp.softplus, dev(dout))
    torch.cuda.synchronize()
    assert tuple(g["dB"].shape) == (bt, G, N, L) and tuple(g["dC"].shape) == (bt, G, N, L)
    bf = dtype == inputs.BF16
    for k in ("du", "ddelta", "dz"):
        grad_close(host_f64(g[k]), ref[k], 1e-4, k, rounded=bf)
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        grad_close(host_f64(g[k]), ref[k], 1e-4, k)
