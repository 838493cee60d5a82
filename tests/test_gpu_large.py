"""The library on activations of more than 2^31 elements.

Three batch rows of 131072 steps x 8192 channels (bf16, d_state 16) make
3.2e9 elements per activation tensor, 6.4 GB each: batch row 2 starts at
element 2^31 and byte 2^32, so every 32-bit element or byte offset would
wrap inside it.  The activations are counter-based draws built on the device
(the host cannot draw 1e10 values in a test's time); the oracle gets the
same values for sampled channels of every batch row, computed on the host
from the same counters.  Checked, on those channels over all steps: the
forward scan's output and final state, the causal conv1d + SiLU, and every
per-channel gradient of the backward.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_out, check_state, dev, host_f64
from selective_state_space_122_b300 import (conv1d_fwd, device_error, inputs, ssm_scan_bwd,
                                            ssm_scan_fwd)

pytestmark = pytest.mark.gpu

BT, L, DIM, N = 3, 131072, 8192, 16
SEED = 2031
STREAM = dict(u=1, delta=2, z=3, dout=4)
# both ends, tile and 32-channel seams, the middle, one random-looking pick
SEL = np.array([0, 1, 31, 32, 4095, 4096, 5003, 8160, 8190, 8191])


def _host_params():
    rng = np.random.Generator(np.random.PCG64(SEED))
    B = inputs._activation(rng, (BT, N, L), inputs.BF16)
    C = inputs._activation(rng, (BT, N, L), inputs.BF16)
    bias = inputs._delta_bias(rng, DIM)
    wconv = (rng.standard_normal((DIM, 4)) * 0.5).astype(np.float32)
    bconv = (rng.standard_normal(DIM) * 0.5).astype(np.float32)
    return B, C, inputs.a_s4d_real(DIM, N), np.ones(DIM, np.float32), bias, wconv, bconv


def _sampled(name):
    return inputs.counter_activation_channels(BT, L, DIM, SEL, STREAM[name], SEED, inputs.BF16)


def _sampled_scan_inputs(B, C, A, D, bias):
    shape = inputs.ScanShape("beyond-2^31 sample", BT, len(SEL), L, N, inputs.BF16)
    return inputs.ScanInputs(shape, _sampled("u"), _sampled("delta"), _sampled("z"), B, C, A[SEL], D[SEL],
                             bias[SEL], True)


@pytest.fixture(scope="module")
def big():
    assert BT * L * DIM > 2**31 and 2 * L * DIM == 2**31
    B, C, A, D, bias, wconv, bconv = _host_params()
    t = {k: inputs.counter_activation_device(BT, L, DIM, STREAM[k], SEED, inputs.BF16, "cuda")
         for k in ("u", "delta", "z")}
    t.update(B=dev(B), C=dev(C), A=dev(A), D=dev(D), bias=dev(bias))
    host = dict(B=B, C=C, A=A, D=D, bias=bias, wconv=wconv, bconv=bconv)
    # the device build holds the host's values (sampled channels, all rows)
    idx = torch.as_tensor(SEL, device="cuda")
    got = t["u"][:, :, idx].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, _sampled("u"))
    yield t, host, idx
    t.clear()
    torch.cuda.empty_cache()


def test_scan_fwd_beyond_2_31_elements(big):
    t, host, idx = big
    out, last = ssm_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["bias"], True,
                             return_last_state=True)
    torch.cuda.synchronize()
    assert device_error() == 0
    f = _sampled_scan_inputs(host["B"], host["C"], host["A"], host["D"], host["bias"]).as_f64()
    ref, ref_last = oracle.scan(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"], f["delta_bias"],
                                f["softplus"])
    for b in range(BT):   # row by row, so a wrap in one row cannot hide behind the others' rms
        check_out(host_f64(out[b:b + 1, :, idx]), ref[b:b + 1], inputs.BF16, f"out, batch row {b}")
        check_state(host_f64(last[b:b + 1, idx]), ref_last[b:b + 1], inputs.BF16, f"last_state, batch row {b}")
        assert bool(torch.isfinite(out[b]).all()), f"non-finite outputs in batch row {b}"


def test_conv1d_beyond_2_31_elements(big):
    t, host, idx = big
    w, bc = host["wconv"], host["bconv"]
    out, _ = conv1d_fwd(t["u"], dev(w), dev(bc), True)
    torch.cuda.synchronize()
    ref, _ = oracle.conv1d(inputs.bf16_bits_to_f64(_sampled("u")), w[SEL], bc[SEL], True, None)
    for b in range(BT):
        check_out(host_f64(out[b:b + 1, :, idx]), ref[b:b + 1], inputs.BF16, f"conv out, batch row {b}")


def test_scan_bwd_beyond_2_31_elements(big):
    t, host, idx = big
    do = inputs.counter_activation_device(BT, L, DIM, STREAM["dout"], SEED, inputs.BF16, "cuda")
    g = ssm_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["bias"], True, do)
    torch.cuda.synchronize()
    assert device_error() == 0
    del do
    f = _sampled_scan_inputs(host["B"], host["C"], host["A"], host["D"], host["bias"]).as_f64()
    ref = oracle.scan_bwd(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"], f["delta_bias"],
                          f["softplus"], inputs.bf16_bits_to_f64(_sampled("dout")))
    for k in ("du", "ddelta", "dz"):
        got = host_f64(g[k][:, :, idx])
        for b in range(BT):
            _close(got[b], ref[k][b], f"{k}, batch row {b}", rounded=True)
    _close(host_f64(g["dA"][idx]), ref["dA"], "dA")
    for k in ("dD", "ddelta_bias"):
        _close(host_f64(g[k][idx]), ref[k], k)
    for k in ("dB", "dC"):
        assert bool(torch.isfinite(g[k]).all()), k


def _close(got, ref, what, rounded=False):
    """The backward tests' bound: |got - ref| <= 1e-4 * max(rms(ref),
    max|ref| / 50) elementwise, plus the half-ulp 2^-8 |ref| of a bf16
    output when ``rounded``."""
    got = np.asarray(got, dtype=np.float64)
    scale = max(float(np.sqrt(np.mean(ref ** 2))), float(np.max(np.abs(ref))) / 50.0, 1e-30)
    bound = 1e-4 * scale + (2.0 ** -8 * np.abs(ref) if rounded else 0.0)
    excess = np.abs(got - ref) - bound
    assert float(np.max(excess)) <= 0.0, (f"{what}: max|err| {float(np.max(np.abs(got - ref))):.3e}, "
                                          f"bound 1e-4 x {scale:.3e}")
