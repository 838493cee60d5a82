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


def _lowbias32_int(x: int) -> int:
    # the hash written out on Python integers, arbitrary precision, masked
    x ^= x >> 16
    x = (x * 0x7FEB352D) & 0xFFFFFFFF
    x ^= x >> 15
    x = (x * 0x846CA68B) & 0xFFFFFFFF
    return x ^ (x >> 16)


def test_counter_draws_match_the_hash_on_both_libraries():
    """The counter-based draws (activations larger than the host can draw)
    equal the lowbias32 hash written out on Python integers, for indices
    below and beyond 2^31 and 2^32, bit for bit on numpy and on torch, and
    torch's bf16 conversion of them equals the host rounding."""
    idx = np.array([0, 1, 2, 2**31 - 1, 2**31, 2**32 - 1, 2**32, 2**33 + 5, 3 * 131072 * 8192 - 1,
                    12345678901], dtype=np.int64)
    for seed, stream in [(7, 1), (0, 0), (123456789, 3)]:
        key = _lowbias32_int(((seed & 0xFFFFFFFF) * 0x9E3779B9 + stream) & 0xFFFFFFFF)
        ref = [_lowbias32_int((int(i) & 0xFFFFFFFF) ^ _lowbias32_int((int(i) >> 32) ^ key)) for i in idx]
        assert [int(v) for v in inputs.counter_bits(idx, stream, seed)] == ref
        assert [int(v) for v in inputs.counter_bits(torch.from_numpy(idx), stream, seed)] == ref
        a = inputs.counter_uniform_np(idx, stream, seed)
        b = inputs.counter_uniform_torch(torch.from_numpy(idx), stream, seed).numpy()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        assert np.array_equal(a, np.array([(h >> 8) * 2.0 ** -23 - 1.0 for h in ref], dtype=np.float32))
        tb = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(inputs.round_to_bf16_bits(a), tb)


def test_counter_draws_are_uniform_and_distinct_per_stream():
    x = inputs.counter_uniform_np(np.arange(1 << 20, dtype=np.int64), 1, 7)
    assert -1.0 <= float(x.min()) and float(x.max()) < 1.0
    assert abs(float(x.mean())) < 5e-3 and abs(float(x.std()) - 1 / np.sqrt(3.0)) < 5e-3
    y = inputs.counter_uniform_np(np.arange(1 << 20, dtype=np.int64), 2, 7)
    assert abs(float(np.corrcoef(x, y)[0, 1])) < 5e-3


def test_counter_activation_device_equals_host_channels():
    """The slice-by-slice tensor build (run here on the CPU) holds exactly the
    values the host computes for sampled channels, slices of odd length."""
    for dt in (inputs.BF16, inputs.F32):
        d = inputs.counter_activation_device(2, 100, 40, 2, 9, dt, "cpu", rows_per_slice=33)
        sel = [0, 5, 39]
        h = inputs.counter_activation_channels(2, 100, 40, sel, 2, 9, dt)
        got = d[:, :, sel].view(torch.int16).numpy().view(np.uint16) if dt == inputs.BF16 else d[:, :, sel].numpy()
        assert np.array_equal(got, h)
