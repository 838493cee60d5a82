"""ssm_scan_fwd_noalloc: the scan for callers that cannot allocate device memory.

Callers inside a framework whose allocator owns the device memory, or code
that must not allocate in its hot loop, cannot hand ssm_scan_fwd a workspace;
ssm_scan_fwd_noalloc runs the same scan on a fixed scratch array inside the
library instead.  These tests call it through the C ABI and compare it with
ssm_scan_fwd, twice in a row on different inputs (every call reuses the one
array, so the second call must not lean on what the first left there).  Its
refusal of sizes beyond the array is pure host logic, tested in the CPU suite
(test_abi_cpu.py).  This file is collected last on purpose.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from gpu_util import check_out, check_state, dev, host_f64
from selective_state_space_122_b300 import _lib, inputs, ssm_scan_fwd

pytestmark = pytest.mark.gpu


def _noalloc(lib, inp, out, last):
    t = [dev(x) for x in (inp.u, inp.delta, inp.A, inp.B, inp.C, inp.D, inp.z, inp.delta_bias)]
    u, dl, A, B, C, D, z, bias = t
    bt, L, dim = u.shape
    code = lib.ssm_scan_fwd_noalloc(u.data_ptr(), dl.data_ptr(), A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                    D.data_ptr(), z.data_ptr(), bias.data_ptr(), 1, out.data_ptr(),
                                    last.data_ptr(), bt, dim, L, A.shape[1],
                                    _lib.SSM_BF16 if inp.shape.dtype == inputs.BF16 else _lib.SSM_F32,
                                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return code


@pytest.mark.parametrize("shape", [inputs.ScanShape("noalloc-a", 2, 96, 300, 16, inputs.BF16),
                                   inputs.ScanShape("noalloc-b", 3, 40, 77, 8, inputs.F32),
                                   inputs.LAYER_130M],
                         ids=lambda s: s.name)
def test_noalloc_matches_scan_two_calls_in_a_row(shape):
    lib = _lib.load_library()
    # two calls in a row on different seeded inputs: state or flags the first
    # call left in the shared array must not leak into the second's result
    for seed in (91, 92):
        inp = inputs.make_scan_inputs(shape, seed)
        ref_out, ref_last = ssm_scan_fwd(dev(inp.u), dev(inp.delta), dev(inp.A), dev(inp.B), dev(inp.C),
                                         dev(inp.D), dev(inp.z), dev(inp.delta_bias), True, return_last_state=True)
        torch.cuda.synchronize()
        out = torch.full_like(ref_out, float("nan"))
        last = torch.full_like(ref_last, float("nan"))
        assert _noalloc(lib, inp, out, last) == 0
        check_out(host_f64(out), host_f64(ref_out), shape.dtype, f"noalloc out (seed {seed})", rounded_sides=2)
        check_state(host_f64(last), host_f64(ref_last), shape.dtype, f"noalloc last_state (seed {seed})")
