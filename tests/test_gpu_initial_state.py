"""Scans that start from a given state (ssm_scan_fwd_from_state) against the
float64 oracle, on every kernel path; prefill in pieces; resume in place."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_out, check_state, dev, host_f64, paths, scan_layout
from selective_state_space_122_b300 import device_error, inputs, ssm_scan_fwd

pytestmark = pytest.mark.gpu


def _h0(bt, dim, N, seed):
    return (np.random.Generator(np.random.PCG64(seed)).standard_normal((bt, dim, N)) * 0.5).astype(np.float32)


def _oracle(inp, h0, lo=0, hi=None, channels=None):
    f = (inp if channels is None else inp.channels(channels)).as_f64()
    hi = f["u"].shape[1] if hi is None else hi
    cut = lambda a, ax: None if a is None else np.ascontiguousarray(np.take(a, range(lo, hi), axis=ax))
    return oracle.scan(cut(f["u"], 1), cut(f["delta"], 1), f["A"], cut(f["B"], 2), cut(f["C"], 2), f["D"],
                       cut(f["z"], 1), f["delta_bias"], f["softplus"],
                       initial_state=None if h0 is None else h0.astype(np.float64))


def _device(inp):
    return {k: dev(getattr(inp, k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias")}


def _scan(t, softplus, lo, hi, initial_state, last_state=None):
    sl = lambda a: None if a is None else a[:, lo:hi].contiguous()
    sb = lambda a: a[:, :, lo:hi].contiguous()
    out, last = ssm_scan_fwd(sl(t["u"]), sl(t["delta"]), t["A"], sb(t["B"]), sb(t["C"]), t["D"], sl(t["z"]),
                             t["delta_bias"], softplus, last_state=last_state,
                             return_last_state=last_state is None, initial_state=initial_state)
    torch.cuda.synchronize()
    assert device_error() == 0, "a scan kernel reported a timed-out wait"
    return out, last


@pytest.mark.parametrize("bt,dim,L,N,dtype", [(2, 64, 200, 16, inputs.BF16), (2, 72, 77, 16, inputs.BF16),
                                              (2, 48, 130, 8, inputs.BF16), (3, 40, 65, 4, inputs.F32),
                                              (1, 32, 50, 16, inputs.F32), (2, 24, 33, 8, inputs.F32)])
def test_initial_state_every_path(bt, dim, L, N, dtype):
    inp = inputs.make_scan_inputs(inputs.ScanShape("h0", bt, dim, L, N, dtype), 500 + dim + L)
    h0 = _h0(bt, dim, N, 600 + L)
    ref, ref_last = _oracle(inp, h0)
    t = _device(inp)
    for g in paths(N, dim, dtype):
        with scan_layout(g):
            out, last = _scan(t, inp.softplus, 0, L, torch.from_numpy(h0).cuda())
        check_out(host_f64(out), ref, dtype, f"out, path {g}")
        check_state(host_f64(last), ref_last, dtype, f"state, path {g}")


@pytest.mark.parametrize("bt,dim,L,N,dtype,cuts", [
    (2, 256, 1000, 16, inputs.BF16, [333, 600]),
    (1, 5120, 3000, 16, inputs.BF16, [1024, 2047]),
    (2, 96, 500, 8, inputs.BF16, [1, 250]),
    (2, 40, 300, 4, inputs.F32, [77]),
])
def test_prefill_in_pieces_matches_whole(bt, dim, L, N, dtype, cuts):
    """A sequence scanned in pieces, each piece from the previous one's final
    state, against the oracle of the whole sequence (the default path)."""
    inp = inputs.make_scan_inputs(inputs.ScanShape("pieces", bt, dim, L, N, dtype), 700 + L)
    sel = np.arange(0, dim, max(1, dim // 96))
    ref, ref_last = _oracle(inp, None, channels=sel)
    t = _device(inp)
    bounds = [0] + cuts + [L]
    state, outs = None, []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        out, state = _scan(t, inp.softplus, lo, hi, state)
        outs.append(out)
    out = torch.cat(outs, dim=1)
    idx = torch.as_tensor(sel, device=out.device)
    check_out(host_f64(out[:, :, idx]), ref, dtype, "pieces out")
    check_state(host_f64(state[:, idx]), ref_last, dtype, "pieces state")


@pytest.mark.parametrize("g", [None, "seg", 0])
def test_resume_in_place(g):
    """initial_state and last_state the same tensor: the state is read before
    it is overwritten, for every path."""
    bt, dim, L, N = 2, 64, 300, 16
    inp = inputs.make_scan_inputs(inputs.ScanShape("inplace", bt, dim, L, N, inputs.BF16), 901)
    h0 = _h0(bt, dim, N, 902)
    ref, ref_last = _oracle(inp, h0)
    t = _device(inp)
    state = torch.from_numpy(h0).cuda()
    with scan_layout(g):
        out, _ = _scan(t, inp.softplus, 0, L, state, last_state=state)
    check_out(host_f64(out), ref, inputs.BF16, "in-place out")
    check_state(host_f64(state), ref_last, inputs.BF16, "in-place state")


@pytest.mark.parametrize("path", ["tmem2", "ws", "seg"])
def test_initial_state_multisegment(path):
    """Many segments per chain: only each chain's first segment reads the
    initial state; the rest continue from the state handed through the workspace."""
    bt, dim, L, N = 1, 5120, 4096, 16
    inp = inputs.make_scan_inputs(inputs.ScanShape("h0-multi", bt, dim, L, N, inputs.BF16), 950)
    h0 = _h0(bt, dim, N, 951)
    sel = np.arange(3, dim, 61)
    ref, ref_last = _oracle(inp, h0[:, sel], channels=sel)
    t = _device(inp)
    with scan_layout(path):
        out, last = _scan(t, inp.softplus, 0, L, torch.from_numpy(h0).cuda())
    idx = torch.as_tensor(sel, device=out.device)
    check_out(host_f64(out[:, :, idx]), ref, inputs.BF16, f"{path} out")
    check_state(host_f64(last[:, idx]), ref_last, inputs.BF16, f"{path} state")


def test_zero_initial_state_equals_plain_scan():
    """An all-zero initial state gives exactly the plain scan's result."""
    inp = inputs.make_scan_inputs(inputs.ScanShape("zero-h0", 2, 128, 500, 16, inputs.BF16), 960)
    t = _device(inp)
    o1, s1 = _scan(t, inp.softplus, 0, 500, None)
    o2, s2 = _scan(t, inp.softplus, 0, 500, torch.zeros(2, 128, 16, device="cuda"))
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
