"""Stored fixtures and the seeded input generator (CPU only)."""
import os

import numpy as np
import torch

import oracle
from selective_state_space_122_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_reproduces_golden_tiny_f32():
    inp = inputs.make_scan_inputs(inputs.TINY_F32, 0)
    f = inp.as_f64()
    out, last = oracle.scan(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"],
                            f["delta_bias"], f["softplus"])
    ref = np.loadtxt(os.path.join(GOLDEN, "tiny_f32_out.txt"))
    ref_last = np.loadtxt(os.path.join(GOLDEN, "tiny_f32_last_state.txt"))
    assert np.array_equal(out.reshape(-1), ref)
    assert np.array_equal(last.reshape(-1), ref_last)


def test_bf16_rounding_matches_torch_rne():
    r = np.random.Generator(np.random.PCG64(5))
    x = np.concatenate([r.standard_normal(100000).astype(np.float32),
                        np.array([1.0, -1.0, 0.0, 1.00390625, 1.01171875, 3.0e38, 1e-40], np.float32)])
    ours = inputs.round_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = inputs.bf16_bits_to_f64(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_generator_is_seeded_and_shaped():
    a = inputs.make_scan_inputs(inputs.ScanShape("t", 2, 24, 32, 16, inputs.BF16), 7)
    b = inputs.make_scan_inputs(a.shape, 7)
    for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias"):
        assert np.array_equal(getattr(a, k), getattr(b, k)), k
    s = a.shape
    assert a.u.shape == (s.batch, s.seqlen, s.dim) and a.u.dtype == np.uint16
    assert a.B.shape == (s.batch, s.dstate, s.seqlen)
    assert a.A.shape == (s.dim, s.dstate) and np.all(a.A < 0)
    # delta_bias = softplus^-1(dt), dt in [1e-3, 0.1]
    dt = np.logaddexp(0.0, a.delta_bias.astype(np.float64))
    assert dt.min() >= 1e-3 * (1 - 1e-5) and dt.max() <= 0.1 * (1 + 1e-5)


def test_decode_generator():
    d = inputs.make_decode_inputs(inputs.DecodeShape("t", 4, 8, 16, inputs.BF16), 3)
    assert d.state0.shape == (4, 8, 16) and d.state0.dtype == np.float32
    assert 0.05 < float(np.std(d.state0)) < 0.2
    x, dt, z, B, C = d.token()
    assert x.shape == (4, 8) and B.shape == (4, 16) and x.dtype == np.uint16


def test_grouped_draws_keep_the_one_group_stream():
    """ngroups = 1 draws exactly the plain inputs; ngroups > 1 draws B and C as
    (batch, ngroups, N, L) in the same order (u, delta, z, then B, then C), so
    the activations drawn before them are unchanged."""
    shape = inputs.ScanShape("g", 2, 24, 10, 4, inputs.BF16)
    a = inputs.make_scan_inputs(shape, 5)
    b = inputs.make_scan_inputs(shape, 5, ngroups=1)
    for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias"):
        assert np.array_equal(getattr(a, k), getattr(b, k)), k
    g = inputs.make_scan_inputs(shape, 5, ngroups=3)
    assert g.B.shape == (2, 3, 4, 10) and g.C.shape == (2, 3, 4, 10)
    for k in ("u", "delta", "z"):
        assert np.array_equal(getattr(a, k), getattr(g, k)), k
    d = inputs.make_decode_inputs(inputs.DecodeShape("g", 3, 8, 4, inputs.F32), 9)
    x, dt, z, B, C = d.token(ngroups=2)
    assert B.shape == (3, 2, 4) and C.shape == (3, 2, 4) and x.shape == (3, 8)
