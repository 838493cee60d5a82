"""Helpers shared by the GPU parity tests: device upload and the tolerances.

Tolerances (from the stated parity bar):
* float32 activations: |err| <= 1e-5 * (1 + |y_ref|) elementwise;
* bf16 activations:    |err| <= 2e-2 * rms(y_ref) + 2^-8 * |y_ref| elementwise,
                       and the final state's relative L2 error <= 1e-3.

The bf16 output bound adds the output format's own rounding to the stated
2e-2 * rms(y_ref): out is stored in the activation dtype, and bf16
round-to-nearest-even moves a value by up to half an ulp, 2^-8 * |y|.  On
these inputs |y| reaches ~50 * rms(y) (y carries D*u*silu(z), a product of
Gaussians), where that rounding alone exceeds 2e-2 * rms(y).
"""
from __future__ import annotations

import contextlib

import numpy as np
import torch

from selective_state_space_122_b300 import inputs

F32_REL = 1e-5
BF16_RMS = 2e-2
BF16_HALF_ULP = 2.0 ** -8
STATE_REL = 1e-3


def dev(a: np.ndarray, dtype: str = None) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def scan_on_gpu(inp: inputs.ScanInputs, want_state=True):
    from selective_state_space_122_b300 import device_error, ssm_scan_fwd
    u, dl, z, B, C = (dev(x) for x in (inp.u, inp.delta, inp.z, inp.B, inp.C))
    out, last = ssm_scan_fwd(u, dl, dev(inp.A), B, C, dev(inp.D), z, dev(inp.delta_bias),
                             inp.softplus, return_last_state=want_state)
    torch.cuda.synchronize()
    assert device_error() == 0, "a scan kernel reported a timed-out wait"
    return out, last


def check_out(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "out", rounded_sides: int = 1):
    """rounded_sides = 2 when ``ref`` is itself a bf16-rounded output (GPU vs GPU):
    two rounded values may then differ by a full ulp, 2 * 2^-8 * |y|."""
    err = np.abs(got - ref)
    if dtype == inputs.F32:
        bound = F32_REL * (1.0 + np.abs(ref))
        bad = err > bound
        assert not bad.any(), (f"{what}: {int(bad.sum())} elements over 1e-5*(1+|y|); "
                               f"worst err {float(err.max()):.3e}")
    else:
        rms = float(np.sqrt(np.mean(ref * ref)))
        excess = err - rounded_sides * BF16_HALF_ULP * np.abs(ref)
        assert float(excess.max()) <= BF16_RMS * rms, (
            f"{what}: max(|err| - 2^-8|y|) {float(excess.max()):.4e} > 2e-2 * rms {rms:.4e} "
            f"(max|err| {float(err.max()):.4e})")
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"


def state_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm((got - ref).ravel()) / np.linalg.norm(ref.ravel()))


def check_state(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "last_state"):
    if dtype == inputs.F32:
        check_out(got, ref, dtype, what)
    else:
        rel = state_rel_err(got, ref)
        assert rel <= STATE_REL, f"{what}: relative L2 error {rel:.3e} > 1e-3"


# number of compiled generic-kernel layouts per d_state (selectable with ssm_force_scan_path)
LAYOUTS = {16: 7, 8: 4, 4: 2}


def tma_rows_ok(dim: int, dtype: str) -> bool:
    """Whether the TMA paths (segmented, tensor-memory) accept this channel
    count: rows of dim elements must be a multiple of 16 bytes for the
    tensor maps."""
    return (dim * (2 if dtype == inputs.BF16 else 4)) % 16 == 0


def tmem_ok(N: int, dim: int, dtype: str) -> bool:
    """Whether the tensor-memory path takes the shape: bf16, 16 states, TMA rows."""
    return N == 16 and dtype == inputs.BF16 and tma_rows_ok(dim, dtype)


def paths(N: int, dim: int = 64, dtype: str = inputs.BF16):
    """Every way to run a scan of this shape: the tensor-memory and segmented
    paths (when they accept the shape) and each generic layout."""
    fast = ["seg"] if tma_rows_ok(dim, dtype) else []
    if tmem_ok(N, dim, dtype):
        fast = ["tmem2", "ws"] + fast
    return fast + list(range(LAYOUTS[N]))


@contextlib.contextmanager
def scan_layout(layout):
    """Force a path (ssm_force_scan_path): None = the library's own choice,
    "tmem2" / "ws" / "seg" = that TMA kernel (an error if it cannot take the
    shape), an int = that layout of the generic kernel."""
    from selective_state_space_122_b300 import force_scan_path
    if layout is None:
        force_scan_path(None)
    elif isinstance(layout, str):
        force_scan_path(layout)
    else:
        force_scan_path("generic", layout)
    try:
        yield
    finally:
        force_scan_path(None)
