"""GPU parity of ssm_state_update (decode) against the oracle and against the scan."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_out, check_state, dev, host_f64
from selective_state_space_122_b300 import inputs, ssm_scan_fwd, ssm_state_update

pytestmark = pytest.mark.gpu


def f64(a, dtype):
    return inputs.bf16_bits_to_f64(a) if dtype == inputs.BF16 else a.astype(np.float64)


def one_step_case(shape, seed, **kw):
    d = inputs.make_decode_inputs(shape, seed)
    x, dt, z, B, C = d.token()
    return d, x, dt, z, B, C


@pytest.mark.parametrize("dtype,N,bt,dim", [(inputs.BF16, 16, 256, 5120), (inputs.F32, 16, 3, 77),
                                             (inputs.BF16, 8, 5, 33), (inputs.F32, 4, 2, 9),
                                             (inputs.BF16, 4, 1, 1),
                                             # enough (row, 128-channel tile) pairs for the
                                             # bulk-copy pipeline; ragged last tiles
                                             (inputs.BF16, 16, 160, 200), (inputs.F32, 16, 300, 132),
                                             (inputs.BF16, 8, 200, 264), (inputs.F32, 4, 400, 136),
                                             (inputs.BF16, 4, 1000, 48)])
def test_single_step_vs_oracle(dtype, N, bt, dim):
    shape = inputs.DecodeShape("step", bt, dim, N, dtype)
    d, x, dt, z, B, C = one_step_case(shape, 4)
    state = dev(d.state0.copy())
    out = ssm_state_update(state, dev(x), dev(dt), dev(d.A), dev(B), dev(C), dev(d.D), dev(z),
                           dev(d.dt_bias), True)
    torch.cuda.synchronize()
    ref_state = d.state0.astype(np.float64)
    ref = oracle.step(ref_state, f64(x, dtype), f64(dt, dtype), d.A, f64(B, dtype), f64(C, dtype),
                      d.D, f64(z, dtype), d.dt_bias, True)
    check_out(host_f64(out), ref, dtype)
    check_state(host_f64(state), ref_state, dtype, "state")


@pytest.mark.parametrize("opts", [dict(softplus=False), dict(no_z=True), dict(no_d=True),
                                  dict(no_bias=True)], ids=["no-softplus", "no-gate", "no-D", "no-bias"])
def test_step_options(opts):
    dtype = inputs.BF16
    shape = inputs.DecodeShape("opts", 4, 96, 16, dtype)
    d, x, dt, z, B, C = one_step_case(shape, 5)
    sp = opts.get("softplus", True)
    bias = None if opts.get("no_bias") else d.dt_bias
    if not sp:
        dt = inputs.round_to_bf16_bits((np.abs(f64(dt, dtype)) * 0.05).astype(np.float32))
        bias = None
    zz = None if opts.get("no_z") else z
    Dd = None if opts.get("no_d") else d.D
    state = dev(d.state0.copy())
    out = ssm_state_update(state, dev(x), dev(dt), dev(d.A), dev(B), dev(C), dev(Dd), dev(zz),
                           dev(bias), sp)
    torch.cuda.synchronize()
    ref_state = d.state0.astype(np.float64)
    ref = oracle.step(ref_state, f64(x, dtype), f64(dt, dtype), d.A, f64(B, dtype), f64(C, dtype),
                      Dd, None if zz is None else f64(zz, dtype), bias, sp)
    check_out(host_f64(out), ref, dtype)
    check_state(host_f64(state), ref_state, dtype, "state")


def test_decode_chain_1000_steps_equals_scan():
    """1000 chained decode steps from a zero state at 256 x 5120 x 16 against
    ssm_scan_fwd over the same 1000 tokens, and both against the oracle on
    sampled rows."""
    shape = inputs.DECODE_256
    steps = 1000
    d = inputs.make_decode_inputs(shape, 6)
    bt, dim, N = shape.batch, shape.dim, shape.dstate
    xs = np.empty((bt, steps, dim), np.uint16)           # scan layout (bt, L, dim)
    dts = np.empty_like(xs)
    zs = np.empty_like(xs)
    Bs = np.empty((bt, N, steps), np.uint16)             # (bt, N, L)
    Cs = np.empty_like(Bs)
    for t in range(steps):
        xs[:, t], dts[:, t], zs[:, t], Bs[:, :, t], Cs[:, :, t] = d.token()

    A, Dv, bias = dev(d.A), dev(d.D), dev(d.dt_bias)
    gx, gdt, gz, gB, gC = dev(xs), dev(dts), dev(zs), dev(Bs), dev(Cs)
    scan_out, scan_state = ssm_scan_fwd(gx, gdt, A, gB, gC, Dv, gz, bias, True, return_last_state=True)

    state = torch.zeros((bt, dim, N), dtype=torch.float32, device="cuda")
    dec_out = torch.empty_like(gx)
    gBt = gB.permute(0, 2, 1).contiguous()               # (bt, L, N)
    gCt = gC.permute(0, 2, 1).contiguous()
    for t in range(steps):
        dec_out[:, t] = ssm_state_update(state, gx[:, t].contiguous(), gdt[:, t].contiguous(), A,
                                         gBt[:, t].contiguous(), gCt[:, t].contiguous(), Dv,
                                         gz[:, t].contiguous(), bias, True)
    torch.cuda.synchronize()

    # both against the oracle on sampled batch rows (all channels)
    rows = np.array([0, 97, 255])
    f = lambda a: np.ascontiguousarray(inputs.bf16_bits_to_f64(a[rows]))
    ref, ref_state = oracle.scan(f(xs), f(dts), d.A, f(Bs), f(Cs), d.D, f(zs), d.dt_bias, True)
    r = torch.as_tensor(rows, device="cuda")
    check_out(host_f64(dec_out[r]), ref, inputs.BF16, "decode vs oracle")
    check_out(host_f64(scan_out[r]), ref, inputs.BF16, "scan vs oracle")
    check_state(host_f64(state[r]), ref_state, inputs.BF16, "decode state vs oracle")
    check_state(host_f64(scan_state[r]), ref_state, inputs.BF16, "scan state vs oracle")

    # decode chain vs scan everywhere (two float32 recurrences, both outputs bf16-rounded)
    check_out(host_f64(dec_out), host_f64(scan_out), inputs.BF16, "decode vs scan out", rounded_sides=2)
    check_state(host_f64(state), host_f64(scan_state), inputs.BF16, "decode vs scan state")


def test_decode_writes_stay_in_bounds():
    shape = inputs.DecodeShape("guard", 3, 50, 16, inputs.BF16)
    d, x, dt, z, B, C = one_step_case(shape, 8)
    guard = 2048
    n = 3 * 50
    buf = torch.full((n + 2 * guard,), 77.0, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + n].view(3, 50)
    sbuf = torch.full((3 * 50 * 16 + 2 * guard,), 5.0, dtype=torch.float32, device="cuda")
    state = sbuf[guard:guard + 3 * 50 * 16].view(3, 50, 16)
    state.copy_(torch.from_numpy(d.state0))
    ssm_state_update(state, dev(x), dev(dt), dev(d.A), dev(B), dev(C), dev(d.D), dev(z), dev(d.dt_bias),
                     True, out=out)
    torch.cuda.synchronize()
    assert bool((buf[:guard] == 77.0).all()) and bool((buf[guard + n:] == 77.0).all())
    assert bool((sbuf[:guard] == 5.0).all()) and bool((sbuf[guard + 3 * 50 * 16:] == 5.0).all())


def test_decode_bulk_writes_stay_in_bounds():
    """The bulk-copy pipeline (160 rows x two 128-channel tiles, the second
    ragged) writes no state or output outside its tensors."""
    bt, dim, N = 160, 200, 16
    shape = inputs.DecodeShape("guard-bulk", bt, dim, N, inputs.BF16)
    d, x, dt, z, B, C = one_step_case(shape, 9)
    guard = 4096
    n = bt * dim
    buf = torch.full((n + 2 * guard,), 77.0, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + n].view(bt, dim)
    sbuf = torch.full((n * N + 2 * guard,), 5.0, dtype=torch.float32, device="cuda")
    state = sbuf[guard:guard + n * N].view(bt, dim, N)
    state.copy_(torch.from_numpy(d.state0))
    ssm_state_update(state, dev(x), dev(dt), dev(d.A), dev(B), dev(C), dev(d.D), dev(z), dev(d.dt_bias),
                     True, out=out)
    torch.cuda.synchronize()
    assert bool((buf[:guard] == 77.0).all()) and bool((buf[guard + n:] == 77.0).all())
    assert bool((sbuf[:guard] == 5.0).all()) and bool((sbuf[guard + n * N:] == 5.0).all())
    ref_state = d.state0.astype(np.float64)
    ref = oracle.step(ref_state, f64(x, inputs.BF16), f64(dt, inputs.BF16), d.A, f64(B, inputs.BF16),
                      f64(C, inputs.BF16), d.D, f64(z, inputs.BF16), d.dt_bias, True)
    check_out(host_f64(out), ref, inputs.BF16)
    check_state(host_f64(state), ref_state, inputs.BF16, "state")
