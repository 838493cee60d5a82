"""The kernels' bounded waits, made to give up on purpose (no fault).

Every wait in the library's kernels is bounded: on running out it sets a bit
in the device error word, and its CTA still drains its copies and frees its
tensor memory before returning.  The wait test hook (ssm_debug_wait_test)
shortens the limit to 2 ms and makes the first segment of channel group 0
keep its hand-off flag unset, so the segment after it waits for a flag that
nothing sets.  The call must come back with bit 4 set; then, with the
defaults restored, the very same scan must be correct -- which it could not
be if tensor memory had leaked or copies had been left in flight.
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_out, check_state, dev, host_f64, scan_layout, scan_on_gpu
from selective_state_space_122_b300 import _lib, device_error, inputs, ssm_scan_fwd, ssm_state_update

pytestmark = pytest.mark.gpu

# 160 groups of 32 channels (640 of 8) for 148 SMs: every chain is cut into
# segments handed from CTA to CTA (warp to warp for the segmented kernel)
SHAPE = inputs.ScanShape("wait-test", 1, 5120, 4096, 16, inputs.BF16)


@pytest.mark.parametrize("path", ["tmem2", "ws", "seg"])
def test_wait_gives_up_then_next_scan_is_correct(path):
    lib = _lib.load_library()
    inp = inputs.make_scan_inputs(SHAPE, 1234)
    t = [dev(x) for x in (inp.u, inp.delta, inp.A, inp.B, inp.C, inp.D, inp.z, inp.delta_bias)]
    torch.cuda.synchronize()
    device_error(clear=True)
    try:
        assert lib.ssm_debug_wait_test(1, 2_000_000) == 0
        with scan_layout(path):
            t0 = time.time()
            ssm_scan_fwd(*t, True, return_last_state=True)
            torch.cuda.synchronize()
            took = time.time() - t0
        err = device_error(clear=True)
    finally:
        assert lib.ssm_debug_wait_test(0, 0) == 0
    assert err & 4, f"no segment hand-off timeout reported (error word {err})"
    assert took < 30.0, f"the call took {took:.1f} s to give up"

    with scan_layout(path):
        out, last = scan_on_gpu(inp)     # also asserts the error word stayed 0
    sel = np.array([0, 1, 17, 31, 32, 500, 2047, 4096, 5119])
    f = inp.channels(sel).as_f64()
    ref, ref_last = oracle.scan(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"], f["delta_bias"], True)
    idx = torch.as_tensor(sel, device=out.device)
    check_out(host_f64(out[:, :, idx]), ref, inputs.BF16)
    check_state(host_f64(last[:, idx]), ref_last, inputs.BF16)


def test_decode_bulk_wait_gives_up_then_next_step_is_correct():
    """The decode step's bulk-copy pipeline: with the hook set, block 0 never
    issues its first row's copies, its consumers wait that stage out (2 ms)
    and give up (bit 1), its producer waits (bounded) for what it issued and
    returns; the next step, with the defaults restored, matches the oracle."""
    lib = _lib.load_library()
    shape = inputs.DecodeShape("wait-decode", 256, 5120, 16, inputs.BF16)
    d = inputs.make_decode_inputs(shape, 77)
    x, dt, z, B, C = d.token()
    args = [dev(x), dev(dt), dev(d.A), dev(B), dev(C), dev(d.D), dev(z), dev(d.dt_bias)]
    state = dev(d.state0.copy())
    torch.cuda.synchronize()
    device_error(clear=True)
    try:
        assert lib.ssm_debug_wait_test(1, 2_000_000) == 0
        t0 = time.time()
        ssm_state_update(state, args[0], args[1], args[2], args[3], args[4], args[5], args[6], args[7], True)
        torch.cuda.synchronize()
        took = time.time() - t0
        err = device_error(clear=True)
    finally:
        assert lib.ssm_debug_wait_test(0, 0) == 0
    assert err & 1, f"no staged-data timeout reported (error word {err})"
    assert took < 30.0, f"the step took {took:.1f} s to give up"

    state = dev(d.state0.copy())
    out = ssm_state_update(state, args[0], args[1], args[2], args[3], args[4], args[5], args[6], args[7], True)
    torch.cuda.synchronize()
    assert device_error(clear=True) == 0
    f = lambda a: inputs.bf16_bits_to_f64(a)
    ref_state = d.state0.astype(np.float64)
    ref = oracle.step(ref_state, f(x), f(dt), d.A, f(B), f(C), d.D, f(z), d.dt_bias, True)
    check_out(host_f64(out), ref, inputs.BF16)
    check_state(host_f64(state), ref_state, inputs.BF16, "state")
