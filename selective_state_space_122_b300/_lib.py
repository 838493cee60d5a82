"""ctypes binding of libssmscan.so (include/ssm_scan.h).

Argument marshalling only: every step of the scan and of the decode update
runs in the library's CUDA kernels.  PyTorch provides device memory and the
current stream.  There is no CPU path: if the library is missing or no CUDA
device is present the calls raise.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional, Tuple

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libssmscan.so")

SSM_F32 = 0
SSM_BF16 = 1
STATUS = {0: "SSM_OK", 1: "SSM_ERR_NULL", 2: "SSM_ERR_SHAPE", 3: "SSM_ERR_ALIGN",
          4: "SSM_ERR_UNSUPPORTED", 5: "SSM_ERR_DTYPE", 6: "SSM_ERR_ALIAS",
          7: "SSM_ERR_LAUNCH", 8: "SSM_ERR_DEVICE", 9: "SSM_ERR_SCRATCH"}
EXPORTS = ("ssm_scan_fwd", "ssm_scan_workspace_bytes", "ssm_device_error", "ssm_state_update",
           "ssm_status_string", "ssm_last_launch_error", "ssm_version", "ssm_scan_fwd_noalloc",
           "ssm_scan_noalloc_max_workspace_bytes", "ssm_scan_fwd_from_state", "ssm_conv1d_fwd",
           "ssm_conv1d_update", "ssm_scan_bwd", "ssm_scan_bwd_workspace_bytes", "ssm_scan_fwd_grouped",
           "ssm_scan_workspace_bytes_grouped", "ssm_state_update_grouped", "ssm_scan_bwd_grouped",
           "ssm_scan_bwd_from_state", "ssm_force_scan_path", "ssm_debug_wait_test")

_lib: Optional[ctypes.CDLL] = None


class SSMError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libssmscan.so and declare its signatures.  Raises if it is absent."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m selective_state_space_122_b300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    vp, fp, i64, ci = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.ssm_scan_fwd.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, vp, fp,
                                 i64, i64, i64, i64, ci, vp, i64, vp]
    lib.ssm_scan_fwd.restype = ci
    lib.ssm_scan_fwd_from_state.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, fp, vp, fp,
                                            i64, i64, i64, i64, ci, vp, i64, vp]
    lib.ssm_scan_fwd_from_state.restype = ci
    lib.ssm_scan_bwd.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, vp, vp, vp, fp, fp, fp, fp, vp, fp,
                                 i64, i64, i64, i64, ci, vp, i64, vp]
    lib.ssm_scan_bwd.restype = ci
    lib.ssm_scan_fwd_grouped.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, fp, vp, fp,
                                         i64, i64, i64, i64, i64, ci, vp, i64, vp]
    lib.ssm_scan_fwd_grouped.restype = ci
    lib.ssm_scan_workspace_bytes_grouped.argtypes = [i64, i64, i64, i64, i64, ci]
    lib.ssm_scan_workspace_bytes_grouped.restype = i64
    lib.ssm_scan_bwd_grouped.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, vp, vp, vp, fp, fp, fp, fp, vp, fp,
                                         i64, i64, i64, i64, i64, ci, vp, i64, vp]
    lib.ssm_scan_bwd_grouped.restype = ci
    lib.ssm_scan_bwd_from_state.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, fp, vp, fp, vp, vp, fp, fp, fp, fp,
                                            vp, fp, fp, i64, i64, i64, i64, i64, ci, vp, i64, vp]
    lib.ssm_scan_bwd_from_state.restype = ci
    lib.ssm_state_update_grouped.argtypes = [fp, vp, vp, fp, vp, vp, fp, vp, fp, vp,
                                             i64, i64, i64, i64, ci, ci, vp]
    lib.ssm_state_update_grouped.restype = ci
    lib.ssm_scan_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64, ci]
    lib.ssm_scan_bwd_workspace_bytes.restype = i64
    lib.ssm_conv1d_fwd.argtypes = [vp, fp, fp, ci, fp, vp, fp, i64, i64, i64, i64, ci, vp]
    lib.ssm_conv1d_fwd.restype = ci
    lib.ssm_conv1d_update.argtypes = [fp, vp, fp, fp, ci, vp, i64, i64, i64, ci, vp]
    lib.ssm_conv1d_update.restype = ci
    lib.ssm_scan_workspace_bytes.argtypes = [i64, i64, i64, i64, ci]
    lib.ssm_scan_workspace_bytes.restype = i64
    lib.ssm_device_error.argtypes = [ci]
    lib.ssm_device_error.restype = ci
    lib.ssm_state_update.argtypes = [fp, vp, vp, fp, vp, vp, fp, vp, fp, vp,
                                     i64, i64, i64, ci, ci, vp]
    lib.ssm_state_update.restype = ci
    lib.ssm_status_string.argtypes = [ci]
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_scan_fwd_noalloc.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, vp, fp,
                                         i64, i64, i64, i64, ci, vp]
    lib.ssm_scan_fwd_noalloc.restype = ci
    lib.ssm_scan_noalloc_max_workspace_bytes.argtypes = []
    lib.ssm_scan_noalloc_max_workspace_bytes.restype = i64
    lib.ssm_last_launch_error.argtypes = []
    lib.ssm_last_launch_error.restype = ctypes.c_char_p
    lib.ssm_version.argtypes = []
    lib.ssm_version.restype = ci
    lib.ssm_force_scan_path.argtypes = [ci, ci]
    lib.ssm_force_scan_path.restype = ci
    lib.ssm_debug_wait_test.argtypes = [ci, i64]
    lib.ssm_debug_wait_test.restype = ci
    if path == LIB_PATH:
        _lib = lib
    return lib


SCAN_PATHS = {None: 0, "tmem2": 1, "ws": 2, "seg": 3, "generic": 4}


def force_scan_path(path: Optional[str] = None, generic_layout: int = -1) -> None:
    """Diagnostics: make every later scan call run one kernel (ssm_force_scan_path).
    path: None (the library's own choice), "tmem2", "ws", "seg" or "generic"."""
    _check("ssm_force_scan_path", load_library().ssm_force_scan_path(SCAN_PATHS[path], int(generic_layout)))


def status_string(code: int) -> str:
    return load_library().ssm_status_string(int(code)).decode()


def _check(fn: str, code: int) -> None:
    if code != 0:
        msg = status_string(code)
        if code == 7:   # SSM_ERR_LAUNCH: add the CUDA runtime's own message
            msg += f" [{load_library().ssm_last_launch_error().decode()}]"
        raise SSMError(fn, code, msg)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    if t.dtype == torch.float32:
        return SSM_F32
    raise TypeError(f"activations must be float32 or bfloat16, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor], dtype=None, device=None) -> Optional[int]:
    if t is None:
        return None
    idx = t.get_device()          # -1 off the GPU; an int compare, cheaper than torch.device objects
    if idx < 0:
        raise ValueError("every tensor must be on a CUDA device")
    if device is not None and idx != device.index:
        raise ValueError("every tensor must be on the same CUDA device")
    if not t.is_contiguous():
        raise ValueError("every tensor must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _on(device: torch.device):
    """The device context of a call: switch only when the tensors live on a
    device other than the current one (the switch costs more than the check)."""
    if device.index is None or device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def scan_workspace_bytes(batch: int, dim: int, seqlen: int, dstate: int, dtype: torch.dtype,
                         ngroups: int = 1) -> int:
    """Workspace bytes the fast path of ssm_scan_fwd needs (ssm_scan_workspace_bytes,
    or ssm_scan_workspace_bytes_grouped for B/C with several channel groups)."""
    code = SSM_BF16 if dtype == torch.bfloat16 else SSM_F32
    lib = load_library()
    if ngroups == 1:
        return int(lib.ssm_scan_workspace_bytes(batch, dim, seqlen, dstate, code))
    return int(lib.ssm_scan_workspace_bytes_grouped(batch, dim, seqlen, dstate, ngroups, code))


def _bc_groups(B: torch.Tensor, C: torch.Tensor, lead: tuple, N: int, tail: tuple, fn: str) -> int:
    """Number of channel groups of B and C: shaped lead + (N,) + tail for one
    group, lead + (ngroups, N) + tail for several.  The device buffers are read
    over exactly that extent, so any other shape is rejected here."""
    G = 1 if B.dim() == len(lead) + 1 + len(tail) else int(B.shape[len(lead)]) if B.dim() > len(lead) else 0
    want = (*lead, N, *tail) if B.dim() == len(lead) + 1 + len(tail) else (*lead, G, N, *tail)
    if G <= 0 or tuple(B.shape) != want or tuple(C.shape) != want:
        raise ValueError(f"{fn}: B and C must be {(*lead, N, *tail)} or {(*lead, 'ngroups', N, *tail)}, "
                         f"got {tuple(B.shape)} and {tuple(C.shape)}")
    return G


def device_error(clear: bool = True) -> int:
    """The library's device error word (0 = no kernel reported a problem); synchronises."""
    return int(load_library().ssm_device_error(int(bool(clear))))


def ssm_scan_fwd(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                 C: torch.Tensor, D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                 delta_bias: Optional[torch.Tensor] = None, softplus: bool = True,
                 out: Optional[torch.Tensor] = None, last_state: Optional[torch.Tensor] = None,
                 return_last_state: bool = False,
                 workspace: Optional[torch.Tensor] = None,
                 initial_state: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Selective scan over (batch, L, dim) activations; see ssm_scan.h.

    B, C: (batch, dstate, L), or (batch, ngroups, dstate, L) for B and C per
    channel group (channel d reads group d // (dim // ngroups);
    ssm_scan_fwd_grouped); A: (dim, dstate) f32; D, delta_bias: (dim,) f32.
    Returns (out, last_state); last_state is (batch, dim, dstate) f32 when
    requested (pass a buffer or set return_last_state).  ``workspace`` is a
    uint8 CUDA tensor of at least scan_workspace_bytes(...) bytes; when None
    one is allocated here (through PyTorch's caching allocator).
    ``initial_state`` (batch, dim, dstate) f32 starts the scan from that state
    (ssm_scan_fwd_from_state); it may be the ``last_state`` tensor itself.
    """
    lib = load_library()
    dt = u.dtype
    dev = u.device
    bt, L, dim = u.shape
    N = A.shape[1]
    G = _bc_groups(B, C, (bt,), N, (L,), "ssm_scan_fwd")
    if out is None:
        out = torch.empty_like(u)
    if last_state is None and return_last_state:
        last_state = torch.empty((bt, dim, N), dtype=torch.float32, device=dev)
    if workspace is None:
        nbytes = scan_workspace_bytes(bt, dim, L, N, dt, G)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev) if nbytes > 0 else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if initial_state is not None and tuple(initial_state.shape) != (bt, dim, N):
        raise ValueError(f"initial_state must be {(bt, dim, N)}, got {tuple(initial_state.shape)}")
    with _on(dev):
        if G != 1:
            code = lib.ssm_scan_fwd_grouped(
                _ptr(u, dt, dev), _ptr(delta, dt, dev), _ptr(A, torch.float32, dev), _ptr(B, dt, dev),
                _ptr(C, dt, dev), _ptr(D, torch.float32, dev), _ptr(z, dt, dev),
                _ptr(delta_bias, torch.float32, dev), int(bool(softplus)),
                _ptr(initial_state, torch.float32, dev), _ptr(out, dt, dev),
                _ptr(last_state, torch.float32, dev), bt, dim, L, N, G, _dtype_code(u),
                _ptr(workspace, None, dev), ws_bytes, _stream(dev))
            _check("ssm_scan_fwd_grouped", code)
        elif initial_state is None:
            code = lib.ssm_scan_fwd(_ptr(u, dt, dev), _ptr(delta, dt, dev), _ptr(A, torch.float32, dev),
                                    _ptr(B, dt, dev), _ptr(C, dt, dev), _ptr(D, torch.float32, dev),
                                    _ptr(z, dt, dev), _ptr(delta_bias, torch.float32, dev),
                                    int(bool(softplus)), _ptr(out, dt, dev),
                                    _ptr(last_state, torch.float32, dev), bt, dim, L, N,
                                    _dtype_code(u), _ptr(workspace, None, dev), ws_bytes, _stream(dev))
            _check("ssm_scan_fwd", code)
        else:
            code = lib.ssm_scan_fwd_from_state(
                _ptr(u, dt, dev), _ptr(delta, dt, dev), _ptr(A, torch.float32, dev), _ptr(B, dt, dev),
                _ptr(C, dt, dev), _ptr(D, torch.float32, dev), _ptr(z, dt, dev),
                _ptr(delta_bias, torch.float32, dev), int(bool(softplus)),
                _ptr(initial_state, torch.float32, dev), _ptr(out, dt, dev),
                _ptr(last_state, torch.float32, dev), bt, dim, L, N, _dtype_code(u),
                _ptr(workspace, None, dev), ws_bytes, _stream(dev))
            _check("ssm_scan_fwd_from_state", code)
    return out, last_state


def ssm_scan_bwd(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
                 D: Optional[torch.Tensor], z: Optional[torch.Tensor], delta_bias: Optional[torch.Tensor],
                 softplus: bool, dout: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                 initial_state: Optional[torch.Tensor] = None, dlast: Optional[torch.Tensor] = None) -> dict:
    """Gradients of the scan (from h = 0) given dout; see ssm_scan.h.  Returns a
    dict du, ddelta, dz (activation dtype; dz None without z), dA, dB, dC, dD,
    ddelta_bias (float32; None without D / bias).  B, C may be grouped as in
    ssm_scan_fwd; dB, dC then have their shape (ssm_scan_bwd_grouped).
    ``initial_state`` (the forward's starting state) and ``dlast`` (dL/d
    last_state), both (batch, dim, dstate) f32, make it the backward of the
    scan from a state (ssm_scan_bwd_from_state); the dict then also holds
    ``dinitial_state`` = dL/d initial_state."""
    lib = load_library()
    dt, dev = u.dtype, u.device
    bt, L, dim = u.shape
    N = A.shape[1]
    G = _bc_groups(B, C, (bt,), N, (L,), "ssm_scan_bwd")
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(du=torch.empty_like(u), ddelta=torch.empty_like(u), dz=None if z is None else torch.empty_like(u),
             dA=torch.empty(dim, N, **f32), dB=torch.empty(tuple(B.shape), **f32),
             dC=torch.empty(tuple(C.shape), **f32),
             dD=None if D is None else torch.empty(dim, **f32),
             ddelta_bias=None if delta_bias is None else torch.empty(dim, **f32))
    if workspace is None:
        nbytes = int(lib.ssm_scan_bwd_workspace_bytes(bt, dim, L, N, _dtype_code(u)))
        if nbytes < 0:
            raise ValueError("ssm_scan_bwd: sizes or dtype rejected")
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    if initial_state is not None or dlast is not None:
        for name, t in (("initial_state", initial_state), ("dlast", dlast)):
            if t is not None and tuple(t.shape) != (bt, dim, N):
                raise ValueError(f"ssm_scan_bwd: {name} must be {(bt, dim, N)}, got {tuple(t.shape)}")
        g["dinitial_state"] = torch.empty(bt, dim, N, **f32)
        with _on(dev):
            code = lib.ssm_scan_bwd_from_state(
                _ptr(u, dt, dev), _ptr(delta, dt, dev), _ptr(A, torch.float32, dev), _ptr(B, dt, dev),
                _ptr(C, dt, dev), _ptr(D, torch.float32, dev), _ptr(z, dt, dev),
                _ptr(delta_bias, torch.float32, dev), int(bool(softplus)), _ptr(initial_state, torch.float32, dev),
                _ptr(dout, dt, dev), _ptr(dlast, torch.float32, dev), _ptr(g["du"], dt, dev),
                _ptr(g["ddelta"], dt, dev), _ptr(g["dA"], torch.float32, dev), _ptr(g["dB"], torch.float32, dev),
                _ptr(g["dC"], torch.float32, dev), _ptr(g["dD"], torch.float32, dev), _ptr(g["dz"], dt, dev),
                _ptr(g["ddelta_bias"], torch.float32, dev), _ptr(g["dinitial_state"], torch.float32, dev),
                bt, dim, L, N, G, _dtype_code(u), _ptr(workspace, None, dev), ws_bytes, _stream(dev))
        _check("ssm_scan_bwd_from_state", code)
        return g
    with _on(dev):
        code = lib.ssm_scan_bwd_grouped(
            _ptr(u, dt, dev), _ptr(delta, dt, dev), _ptr(A, torch.float32, dev), _ptr(B, dt, dev),
            _ptr(C, dt, dev), _ptr(D, torch.float32, dev), _ptr(z, dt, dev), _ptr(delta_bias, torch.float32, dev),
            int(bool(softplus)), _ptr(dout, dt, dev), _ptr(g["du"], dt, dev), _ptr(g["ddelta"], dt, dev),
            _ptr(g["dA"], torch.float32, dev), _ptr(g["dB"], torch.float32, dev), _ptr(g["dC"], torch.float32, dev),
            _ptr(g["dD"], torch.float32, dev), _ptr(g["dz"], dt, dev), _ptr(g["ddelta_bias"], torch.float32, dev),
            bt, dim, L, N, G, _dtype_code(u), _ptr(workspace, None, dev), ws_bytes, _stream(dev))
    _check("ssm_scan_bwd_grouped" if G != 1 else "ssm_scan_bwd", code)
    return g


def conv1d_fwd(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor] = None,
               silu: bool = True, state_in: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
               state_out: Optional[torch.Tensor] = None,
               return_state: bool = False) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Depthwise causal conv1d (+ SiLU) over (batch, L, dim); see ssm_scan.h.
    weight: (dim, W) f32; bias: (dim,) f32; state_in / state_out: (batch, dim,
    W-1) f32 (state_out may be state_in).  Returns (out, state_out)."""
    lib = load_library()
    dt, dev = x.dtype, x.device
    bt, L, dim = x.shape
    W = weight.shape[1]
    if out is None:
        out = torch.empty_like(x)
    if state_out is None and return_state:
        state_out = torch.empty((bt, dim, W - 1), dtype=torch.float32, device=dev)
    with _on(dev):
        code = lib.ssm_conv1d_fwd(_ptr(x, dt, dev), _ptr(weight, torch.float32, dev),
                                  _ptr(bias, torch.float32, dev), int(bool(silu)),
                                  _ptr(state_in, torch.float32, dev), _ptr(out, dt, dev),
                                  _ptr(state_out, torch.float32, dev), bt, dim, L, W, _dtype_code(x),
                                  _stream(dev))
    _check("ssm_conv1d_fwd", code)
    return out, state_out


def conv1d_update(state: torch.Tensor, x: torch.Tensor, weight: torch.Tensor,
                  bias: Optional[torch.Tensor] = None, silu: bool = True,
                  out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One decode step of the conv, in place on ``state`` (batch, dim, W-1) f32."""
    lib = load_library()
    dt, dev = x.dtype, x.device
    bt, dim = x.shape
    W = weight.shape[1]
    if out is None:
        out = torch.empty_like(x)
    with _on(dev):
        code = lib.ssm_conv1d_update(_ptr(state, torch.float32, dev), _ptr(x, dt, dev),
                                     _ptr(weight, torch.float32, dev), _ptr(bias, torch.float32, dev),
                                     int(bool(silu)), _ptr(out, dt, dev), bt, dim, W, _dtype_code(x), _stream(dev))
    _check("ssm_conv1d_update", code)
    return out


def ssm_state_update(state: torch.Tensor, x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor,
                     B: torch.Tensor, C: torch.Tensor, D: Optional[torch.Tensor] = None,
                     z: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
                     dt_softplus: bool = True, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One decode step, in place on ``state`` (batch, dim, dstate) f32; see ssm_scan.h.

    x, dt, z: (batch, dim); B, C: (batch, dstate), or (batch, ngroups, dstate)
    for B and C per channel group (ssm_state_update_grouped).  Returns out
    (batch, dim).
    """
    lib = load_library()
    ty = x.dtype
    dev = x.device
    bt, dim, N = state.shape
    G = _bc_groups(B, C, (bt,), N, (), "ssm_state_update")
    if out is None:
        out = torch.empty_like(x)
    with _on(dev):
        code = lib.ssm_state_update_grouped(_ptr(state, torch.float32, dev), _ptr(x, ty, dev), _ptr(dt, ty, dev),
                                            _ptr(A, torch.float32, dev), _ptr(B, ty, dev), _ptr(C, ty, dev),
                                            _ptr(D, torch.float32, dev), _ptr(z, ty, dev),
                                            _ptr(dt_bias, torch.float32, dev), _ptr(out, ty, dev),
                                            bt, dim, N, G, int(bool(dt_softplus)), _dtype_code(x), _stream(dev))
    _check("ssm_state_update_grouped" if G != 1 else "ssm_state_update", code)
    return out
