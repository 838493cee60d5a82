"""The causal conv1d (+ SiLU) and its decode step against the float64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_out, dev, host_f64
from selective_state_space_122_b300 import conv1d_fwd, conv1d_update, inputs

pytestmark = pytest.mark.gpu


def _case(bt, L, dim, W, dtype, seed, with_bias=True, with_state=True):
    """Seeded inputs: x like the scan's activations (N(0,1) rounded to the
    dtype), taps and bias N(0, 0.5), a carried state N(0, 1)."""
    r = np.random.Generator(np.random.PCG64(seed))
    x = inputs._activation(r, (bt, L, dim), dtype)
    w = (r.standard_normal((dim, W)) * 0.5).astype(np.float32)
    bias = (r.standard_normal(dim) * 0.5).astype(np.float32) if with_bias else None
    st = r.standard_normal((bt, dim, W - 1)).astype(np.float32) if with_state else None
    xf = inputs.bf16_bits_to_f64(x) if dtype == inputs.BF16 else x.astype(np.float64)
    return x, w, bias, st, xf


def _check_state(got, ref, what):
    # the state holds inputs copied exactly (bf16 or f32 values widened to f32)
    assert np.array_equal(got.astype(np.float64), ref), what


@pytest.mark.parametrize("dtype", [inputs.BF16, inputs.F32])
@pytest.mark.parametrize("bt,L,dim,W", [(2, 200, 64, 4), (1, 1000, 5120, 4), (3, 77, 24, 3), (2, 65, 40, 2),
                                         (2, 3, 16, 4), (1, 1, 8, 4), (2, 130, 45, 4), (1, 50, 32, 1)])
@pytest.mark.parametrize("silu", [True, False])
def test_conv1d_fwd(bt, L, dim, W, dtype, silu):
    x, w, bias, st, xf = _case(bt, L, dim, W, dtype, 17 * dim + L + W)
    st = st if W > 1 else None
    ref, ref_st = oracle.conv1d(xf, w, bias, silu, st)
    out, got_st = conv1d_fwd(dev(x), dev(w), dev(bias), silu, None if st is None else dev(st),
                             return_state=W > 1)
    torch.cuda.synchronize()
    check_out(host_f64(out), ref, dtype, f"conv out W={W}")
    if W > 1:
        _check_state(host_f64(got_st), ref_st, "conv final state")


@pytest.mark.parametrize("dtype", [inputs.BF16, inputs.F32])
def test_conv1d_pieces_and_in_place_state(dtype):
    """A sequence convolved in pieces, the state carried in place, equals the
    whole; then a chain of decode steps continues it."""
    bt, L, dim, W = 2, 300, 64, 4
    x, w, bias, st, xf = _case(bt, L, dim, W, dtype, 77)
    ref, ref_st = oracle.conv1d(xf, w, bias, True, st)
    xd, wd, bd = dev(x), dev(w), dev(bias)
    state = dev(st).clone()
    outs = []
    for lo, hi in ((0, 1), (1, 2), (2, 130), (130, 300)):
        o, _ = conv1d_fwd(xd[:, lo:hi].contiguous(), wd, bd, True, state, state_out=state)
        outs.append(o)
    torch.cuda.synchronize()
    check_out(host_f64(torch.cat(outs, dim=1)), ref, dtype, "conv pieces")
    _check_state(host_f64(state), ref_st, "conv pieces state")
    # decode continues from the carried state
    r = np.random.Generator(np.random.PCG64(78))
    ost = ref_st.copy()
    for _ in range(5):
        xt = inputs._activation(r, (bt, dim), dtype)
        xt_f = inputs.bf16_bits_to_f64(xt) if dtype == inputs.BF16 else xt.astype(np.float64)
        ro = oracle.conv1d_update(ost, xt_f, w, bias, True)
        go = conv1d_update(state, dev(xt), wd, bd, True)
        torch.cuda.synchronize()
        check_out(host_f64(go), ro, dtype, "conv decode out")
        _check_state(host_f64(state), ost, "conv decode state")


def test_conv1d_long_sequence_sampled():
    """The long-sequence shape (1 x 131072 x 5120, width 4, bf16, SiLU, carried
    state) in one call, against the oracle on sampled channels over every step:
    the kernel's full tile grid and its 16-byte vector path at full size."""
    bt, L, dim, W = 1, 131072, 5120, 4
    r = np.random.Generator(np.random.PCG64(4242))
    x = inputs._activation(r, (bt, L, dim), inputs.BF16)
    w = (r.standard_normal((dim, W)) * 0.5).astype(np.float32)
    bias = (r.standard_normal(dim) * 0.5).astype(np.float32)
    st = r.standard_normal((bt, dim, W - 1)).astype(np.float32)
    out, got_st = conv1d_fwd(dev(x), dev(w), dev(bias), True, dev(st), return_state=True)
    torch.cuda.synchronize()
    sel = np.unique(np.concatenate([np.arange(0, 16), np.arange(2001, dim, 389), np.arange(dim - 9, dim)]))
    xs = inputs.bf16_bits_to_f64(np.ascontiguousarray(x[:, :, sel]))
    ref, ref_st = oracle.conv1d(xs, w[sel], bias[sel], True, st[:, sel].astype(np.float64))
    idx = torch.as_tensor(sel, device=out.device)
    check_out(host_f64(out[:, :, idx]), ref, inputs.BF16, "long conv out")
    _check_state(host_f64(got_st[:, idx]), ref_st, "long conv state")
