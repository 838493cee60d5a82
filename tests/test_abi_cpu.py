"""The C ABI on the host: symbols, status strings and argument validation.

Every call here is rejected by host-side validation before the library touches
a device, so the tests run without a GPU (the pointers are never dereferenced).
"""
import ctypes
import os
import re

import pytest
import torch

from selective_state_space_122_b300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_scan.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_documented_entry_points():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {_lib.LIB_PATH}").read()
    exported = set(re.findall(r" T (ssm_\w+)", out))
    assert exported == set(declared_functions()), exported


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.ssm_status_string(code).decode().startswith(name)
    assert lib.ssm_status_string(99) == b"unknown ssm_status"
    assert lib.ssm_version() >= 100


P = 0x10000000          # fake, suitably aligned device addresses; never dereferenced
MB = 1 << 20


def scan_args(**kw):
    a = dict(u=P, delta=P + 64 * MB, A=P + 128 * MB, B=P + 192 * MB, C=P + 256 * MB, D=P + 320 * MB,
             z=P + 384 * MB, delta_bias=P + 448 * MB, softplus=1, out=P + 512 * MB,
             last_state=P + 576 * MB, batch=2, dim=64, seqlen=128, dstate=16, dtype=1,
             workspace=None, workspace_bytes=0, stream=None)
    a.update(kw)
    return a


def call_scan(lib, a):
    return lib.ssm_scan_fwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                            a["delta_bias"], a["softplus"], a["out"], a["last_state"], a["batch"],
                            a["dim"], a["seqlen"], a["dstate"], a["dtype"], a["workspace"],
                            a["workspace_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(u=None), 1), (dict(delta=None), 1), (dict(A=None), 1), (dict(B=None), 1),
    (dict(C=None), 1), (dict(out=None), 1),
    (dict(batch=0), 2), (dict(dim=0), 2), (dict(seqlen=0), 2), (dict(seqlen=-5), 2),
    (dict(batch=70000), 2), (dict(dim=1 << 24, seqlen=1 << 20), 2),
    (dict(dstate=3), 4), (dict(dstate=32), 4), (dict(dstate=0), 2),
    (dict(dtype=2), 5), (dict(dtype=-1), 5),
    (dict(u=P + 1), 3), (dict(out=P + 512 * MB + 1), 3), (dict(A=P + 128 * MB + 2), 3),
    (dict(dtype=0, z=P + 384 * MB + 2), 3), (dict(last_state=P + 576 * MB + 2), 3),
    (dict(out=P + 1024), 6), (dict(out=P + 256 * MB), 6), (dict(last_state=P + 512 * MB + 64), 6),
    (dict(last_state=P + 128 * MB), 6),
    (dict(workspace=P + 640 * MB, workspace_bytes=-1), 2), (dict(workspace=P + 640 * MB), 2),
    (dict(workspace=P + 640 * MB + 8, workspace_bytes=MB), 3),
    (dict(workspace=P + 1024, workspace_bytes=MB), 6), (dict(workspace=P + 510 * MB, workspace_bytes=4 * MB), 6),
])
def test_scan_rejects_bad_arguments(lib, kw, code):
    assert call_scan(lib, scan_args(**kw)) == code


def call_scan_from(lib, a, h0):
    return lib.ssm_scan_fwd_from_state(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                       a["delta_bias"], a["softplus"], h0, a["out"], a["last_state"],
                                       a["batch"], a["dim"], a["seqlen"], a["dstate"], a["dtype"],
                                       a["workspace"], a["workspace_bytes"], a["stream"])


@pytest.mark.parametrize("h0,code", [
    (P + 704 * MB + 2, 3),             # misaligned
    (P + 512 * MB + 64, 6),            # inside out
    (P + 64 * MB, 6),                  # inside delta (an input)
    (P + 576 * MB + 64, 6),            # overlaps last_state without being it
])
def test_scan_from_state_rejects_bad_initial_state(lib, h0, code):
    assert call_scan_from(lib, scan_args(), h0) == code


def test_scan_from_state_validates_like_scan(lib):
    """Same host checks as ssm_scan_fwd (only argument sets that are rejected
    before anything is enqueued: these addresses are fake)."""
    for kw in (dict(u=None), dict(dstate=3), dict(u=P + 1), dict(out=P + 1024), dict(batch=0)):
        assert call_scan_from(lib, scan_args(**kw), None) == call_scan(lib, scan_args(**kw))
        assert call_scan_from(lib, scan_args(**kw), P + 704 * MB) == call_scan(lib, scan_args(**kw))
    # an initial state inside the workspace
    assert call_scan_from(lib, scan_args(workspace=P + 704 * MB, workspace_bytes=MB), P + 704 * MB) == 6


def call_conv(lib, **kw):
    a = dict(x=P, w=P + 64 * MB, bias=P + 128 * MB, silu=1, st_in=P + 192 * MB, out=P + 256 * MB,
             st_out=P + 320 * MB, batch=2, dim=64, seqlen=128, width=4, dtype=1, stream=None)
    a.update(kw)
    return lib.ssm_conv1d_fwd(a["x"], a["w"], a["bias"], a["silu"], a["st_in"], a["out"], a["st_out"], a["batch"],
                              a["dim"], a["seqlen"], a["width"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), 1), (dict(w=None), 1), (dict(out=None), 1), (dict(seqlen=0), 2), (dict(width=0), 2),
    (dict(width=5), 4), (dict(dtype=3), 5), (dict(x=P + 1), 3), (dict(st_out=P + 320 * MB + 2), 3),
    (dict(out=P + 64), 6), (dict(out=P + 64 * MB), 6), (dict(st_out=P + 8), 6),
    (dict(st_out=P + 192 * MB + 4), 6),
])
def test_conv1d_rejects_bad_arguments(lib, kw, code):
    assert call_conv(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(state=None), 1), (dict(x=None), 1), (dict(width=7), 4), (dict(batch=0), 2),
    (dict(out=P + 8), 6), (dict(state=P + 64 * MB + 4), 6), (dict(state=P + 2), 3),
])
def test_conv1d_update_rejects_bad_arguments(lib, kw, code):
    a = dict(state=P + 192 * MB, x=P, w=P + 64 * MB, bias=P + 128 * MB, silu=1, out=P + 256 * MB,
             batch=2, dim=64, width=4, dtype=1, stream=None)
    a.update(kw)
    assert lib.ssm_conv1d_update(a["state"], a["x"], a["w"], a["bias"], a["silu"], a["out"], a["batch"],
                                 a["dim"], a["width"], a["dtype"], a["stream"]) == code


@pytest.mark.parametrize("kw,code", [
    (dict(ws=None), 1), (dict(du=None), 1), (dict(dstate=3), 4), (dict(seqlen=0), 2), (dict(dtype=7), 5),
    (dict(ws_bytes=16), 2), (dict(du=P), 6), (dict(dA=P + 128 * MB + 4), 6), (dict(ws=P + 1088 * MB + 8), 3),
])
def test_scan_bwd_rejects_bad_arguments(lib, kw, code):
    """Host checks of ssm_scan_bwd (fake addresses; every case is rejected before
    anything is enqueued)."""
    a = dict(u=P, delta=P + 64 * MB, A=P + 128 * MB, B=P + 192 * MB, C=P + 256 * MB, D=P + 320 * MB,
             z=P + 384 * MB, bias=P + 448 * MB, dout=P + 512 * MB, du=P + 576 * MB, dd=P + 640 * MB,
             dA=P + 704 * MB, dB=P + 768 * MB, dC=P + 832 * MB, dD=P + 896 * MB, dz=P + 960 * MB,
             db=P + 1024 * MB, ws=P + 1088 * MB, ws_bytes=64 * MB, batch=2, dim=64, seqlen=128, dstate=16,
             dtype=1)
    a.update(kw)
    assert lib.ssm_scan_bwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], 1, a["dout"],
                            a["du"], a["dd"], a["dA"], a["dB"], a["dC"], a["dD"], a["dz"], a["db"], a["batch"],
                            a["dim"], a["seqlen"], a["dstate"], a["dtype"], a["ws"], a["ws_bytes"], None) == code
    for args in ((2, 64, 128, 16), (1, 37, 1100, 16), (8, 2048, 2048, 16), (1, 5120, 131072, 16),
                 (3, 48, 1, 4)):
        assert lib.ssm_scan_bwd_workspace_bytes(*args, 1) == _bwd_ws_expected(*args), args
        assert lib.ssm_scan_bwd_workspace_bytes(*args, 0) == _bwd_ws_expected(*args), args


def upd_args(**kw):
    a = dict(state=P, x=P + 64 * MB, dt=P + 128 * MB, A=P + 192 * MB, B=P + 256 * MB, C=P + 320 * MB,
             D=P + 384 * MB, z=P + 448 * MB, dt_bias=P + 512 * MB, out=P + 576 * MB,
             batch=4, dim=64, dstate=16, softplus=1, dtype=1, stream=None)
    a.update(kw)
    return a


def call_upd(lib, a):
    return lib.ssm_state_update(a["state"], a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                a["dt_bias"], a["out"], a["batch"], a["dim"], a["dstate"], a["softplus"],
                                a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(state=None), 1), (dict(x=None), 1), (dict(dt=None), 1), (dict(A=None), 1), (dict(out=None), 1),
    (dict(batch=0), 2), (dict(dim=-1), 2), (dict(dstate=12), 4), (dict(dtype=7), 5),
    (dict(state=P + 8), 3), (dict(A=P + 192 * MB + 4), 3), (dict(x=P + 64 * MB + 1), 3),
    (dict(out=P + 64 * MB), 6), (dict(out=P + 100), 6), (dict(x=P + 2048), 6),
])
def test_update_rejects_bad_arguments(lib, kw, code):
    assert call_upd(lib, upd_args(**kw)) == code


@pytest.mark.skipif(torch.cuda.is_available(), reason="valid arguments would launch on a real device")
def test_valid_call_without_device_reports_device_error(lib):
    assert call_scan(lib, scan_args()) == 8
    assert call_upd(lib, upd_args()) == 8
    # the wait test hook writes device memory: without a device it reports so
    assert lib.ssm_debug_wait_test(0, 0) == 8


def test_binding_raises_without_cuda_tensors():
    u = torch.zeros(1, 8, 8)
    A = torch.zeros(8, 4)
    B = torch.zeros(1, 4, 8)
    with pytest.raises(ValueError):
        _lib.ssm_scan_fwd(u, u, A, B, B)


def _bwd_ws_expected(batch, dim, L, N):
    """The backward's workspace as ssm_scan.h documents it: per-chunk local
    states and Delta sums, three per-segment aggregates, each rounded up to
    256 bytes."""
    r = lambda x: (x + 255) // 256 * 256
    nch = (L + 7) // 8
    S = min(64, max(1, (nch + 31) // 32))
    return max(16, r(batch * nch * dim * N * 4) + r(batch * nch * dim * 4) + 3 * r(batch * S * dim * N * 4))


def _ws_expected(batch, dim, seqlen, dstate, es, ngroups=1):
    """The larger of the fast paths' needs, each part rounded up to 256 bytes:
    B and C staged in the activation type (es bytes, sequence padded to 64
    steps) plus one float32 state per (chain, channel, state) and one int flag
    per chain; and, for bf16 with 16 states, the tensor-memory paths' one-hot
    operands (32 float32 per step) plus their state and one flag per consumer
    warp (up to eight) of each 32-channel group.  Staged B/C (and operands)
    are per (batch row, B/C group)."""
    up = lambda x: (x + 255) // 256 * 256
    lpad = (seqlen + 63) // 64 * 64
    cw = 32 // (dstate // 4)
    chains = batch * ((dim + cw - 1) // cw)
    need = up(batch * ngroups * lpad * 2 * dstate * es) + up(chains * cw * dstate * 4) + up(chains * 4)
    if es == 2 and dstate == 16:
        groups = batch * ((dim + 31) // 32)
        need = max(need, up(batch * ngroups * lpad * 32 * 4) + up(groups * 32 * 16 * 4) + up(groups * 8 * 4))
    return need


def test_workspace_size_query(lib):
    for args in [(1, 5120, 131072, 16), (3, 7, 77, 8), (1, 1, 1, 4), (8, 2048, 2048, 16), (2, 100, 33, 8)]:
        assert lib.ssm_scan_workspace_bytes(*args, 1) == _ws_expected(*args, 2), args
        assert lib.ssm_scan_workspace_bytes(*args, 0) == _ws_expected(*args, 4), args
    assert lib.ssm_scan_workspace_bytes(1, 5120, 131072, 16, 0) == 16777216 + 327680 + 2560
    assert lib.ssm_scan_workspace_bytes(1, 5120, 131072, 16, 1) == 16777216 + 327680 + 5120
    assert lib.ssm_scan_workspace_bytes(1, 64, 64, 5, 1) == -1
    assert lib.ssm_scan_workspace_bytes(1, 64, 0, 16, 1) == -1
    assert lib.ssm_scan_workspace_bytes(1, 0, 64, 16, 1) == -1
    assert lib.ssm_scan_workspace_bytes(1, 64, 64, 16, 7) == -1


def test_grouped_workspace_size_query(lib):
    for args, G in [((1, 5120, 8192, 16), 8), ((3, 96, 77, 8), 3), ((2, 64, 100, 4), 64), ((8, 2048, 2048, 16), 1)]:
        for dt, es in ((1, 2), (0, 4)):
            assert lib.ssm_scan_workspace_bytes_grouped(*args, G, dt) == _ws_expected(*args, es, G), (args, G)
        assert lib.ssm_scan_workspace_bytes_grouped(*args, 1, 1) == lib.ssm_scan_workspace_bytes(*args, 1)
    for G in (0, -2, 3, 65):
        assert lib.ssm_scan_workspace_bytes_grouped(2, 64, 128, 16, G, 1) == -1, G


def call_scan_grouped(lib, a, ngroups, h0=None):
    return lib.ssm_scan_fwd_grouped(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                    a["delta_bias"], a["softplus"], h0, a["out"], a["last_state"],
                                    a["batch"], a["dim"], a["seqlen"], a["dstate"], ngroups, a["dtype"],
                                    a["workspace"], a["workspace_bytes"], a["stream"])


@pytest.mark.parametrize("kw,ngroups,code", [
    ({}, 0, 2), ({}, -1, 2), ({}, 3, 2), ({}, 128, 2), (dict(dim=96), 64, 2),
    (dict(u=None), 4, 1), (dict(dstate=3), 4, 4), (dict(dtype=9), 4, 5), (dict(B=P + 192 * MB + 1), 4, 3),
    # out just past B's one-group extent (2*16*128 bf16) but inside its 4-group extent
    (dict(out=P + 192 * MB + 3 * 8192), 4, 6),
    (dict(last_state=P + 256 * MB + 30000), 4, 6),
])
def test_scan_grouped_rejects_bad_arguments(lib, kw, ngroups, code):
    """Host checks of ssm_scan_fwd_grouped: ngroups must divide dim, and B, C
    span batch * ngroups * dstate * seqlen elements (fake addresses; every case
    is rejected before anything is enqueued)."""
    assert call_scan_grouped(lib, scan_args(**kw), ngroups) == code


def test_scan_grouped_one_group_validates_like_scan(lib):
    for kw in (dict(u=None), dict(dstate=3), dict(u=P + 1), dict(out=P + 1024), dict(batch=0)):
        assert call_scan_grouped(lib, scan_args(**kw), 1) == call_scan(lib, scan_args(**kw))


@pytest.mark.parametrize("kw,ngroups,code", [
    ({}, 0, 2), ({}, 5, 2), (dict(x=None), 2, 1), (dict(dstate=12), 2, 4),
    # out just past B's one-group extent (4*16 bf16) but inside its 8-group extent
    (dict(out=P + 256 * MB + 256), 8, 6),
])
def test_update_grouped_rejects_bad_arguments(lib, kw, ngroups, code):
    a = upd_args(**kw)
    assert lib.ssm_state_update_grouped(a["state"], a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                        a["dt_bias"], a["out"], a["batch"], a["dim"], a["dstate"], ngroups,
                                        a["softplus"], a["dtype"], a["stream"]) == code


@pytest.mark.parametrize("kw,ngroups,code", [
    ({}, 0, 2), ({}, 7, 2), (dict(ws=None), 2, 1),
    # dC 512 KB after dB: apart for one group (dB 2*16*128 f32 = 16 KB), overlapping
    # for 64 groups (1 MB)
    (dict(dC=P + 768 * MB + 512 * 1024), 64, 6),
])
def test_scan_bwd_grouped_rejects_bad_arguments(lib, kw, ngroups, code):
    a = dict(u=P, delta=P + 64 * MB, A=P + 128 * MB, B=P + 192 * MB, C=P + 256 * MB, D=P + 320 * MB,
             z=P + 384 * MB, bias=P + 448 * MB, dout=P + 512 * MB, du=P + 576 * MB, dd=P + 640 * MB,
             dA=P + 704 * MB, dB=P + 768 * MB, dC=P + 832 * MB, dD=P + 896 * MB, dz=P + 960 * MB,
             db=P + 1024 * MB, ws=P + 1088 * MB, ws_bytes=64 * MB, batch=2, dim=64, seqlen=128, dstate=16,
             dtype=1)
    a.update(kw)
    assert lib.ssm_scan_bwd_grouped(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], 1,
                                    a["dout"], a["du"], a["dd"], a["dA"], a["dB"], a["dC"], a["dD"], a["dz"],
                                    a["db"], a["batch"], a["dim"], a["seqlen"], a["dstate"], ngroups, a["dtype"],
                                    a["ws"], a["ws_bytes"], None) == code


def test_binding_checks_bc_shapes():
    """The binding rejects B / C whose shape is neither (batch, N, L) nor
    (batch, ngroups, N, L) before anything reaches the library."""
    u = torch.zeros(2, 8, 8)
    A = torch.zeros(8, 4)
    for B in (torch.zeros(2, 4, 9), torch.zeros(2, 2, 3, 8), torch.zeros(1, 4, 8)):
        with pytest.raises(ValueError, match="B and C must be"):
            _lib.ssm_scan_fwd(u, u, A, B, B)
    st = torch.zeros(2, 8, 4)
    with pytest.raises(ValueError, match="B and C must be"):
        _lib.ssm_state_update(st, u[:, 0], u[:, 0], A, torch.zeros(2, 2, 5), torch.zeros(2, 2, 5))


@pytest.mark.parametrize("kw,code", [
    (dict(h0=P + 1200 * MB + 4), 3), (dict(dlast=P + 1264 * MB + 8), 3), (dict(dh0=P + 1328 * MB + 4), 3),
    (dict(dh0=P + 704 * MB), 6),                  # the initial-state gradient inside dA
    (dict(dh0=P + 1200 * MB), 6),                 # ... over the initial state (an input)
    (dict(h0=P + 576 * MB), 6),                   # the initial state inside du (an output)
    (dict(dlast=P + 640 * MB + 64), 6),           # dlast inside ddelta
    (dict(ngroups=3), 2), (dict(du=None), 1),
])
def test_scan_bwd_from_state_rejects_bad_arguments(lib, kw, code):
    """Host checks of ssm_scan_bwd_from_state (fake addresses; every case is
    rejected before anything is enqueued)."""
    a = dict(u=P, delta=P + 64 * MB, A=P + 128 * MB, B=P + 192 * MB, C=P + 256 * MB, D=P + 320 * MB,
             z=P + 384 * MB, bias=P + 448 * MB, dout=P + 512 * MB, du=P + 576 * MB, dd=P + 640 * MB,
             dA=P + 704 * MB, dB=P + 768 * MB, dC=P + 832 * MB, dD=P + 896 * MB, dz=P + 960 * MB,
             db=P + 1024 * MB, ws=P + 1088 * MB, ws_bytes=64 * MB, h0=P + 1200 * MB, dlast=P + 1264 * MB,
             dh0=P + 1328 * MB, batch=2, dim=64, seqlen=128, dstate=16, ngroups=1, dtype=1)
    a.update(kw)
    assert lib.ssm_scan_bwd_from_state(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], 1,
                                       a["h0"], a["dout"], a["dlast"], a["du"], a["dd"], a["dA"], a["dB"], a["dC"],
                                       a["dD"], a["dz"], a["db"], a["dh0"], a["batch"], a["dim"], a["seqlen"],
                                       a["dstate"], a["ngroups"], a["dtype"], a["ws"], a["ws_bytes"], None) == code


def test_size_products_that_overflow_64_bits_are_rejected(lib):
    """batch * seqlen * dim (or batch * dim) beyond 64 bits must not wrap into
    an accepted size: every such call is SSM_ERR_SHAPE before anything else."""
    big = dict(batch=1, seqlen=1 << 40, dim=1 << 30)     # 2^70 elements
    assert call_scan(lib, scan_args(**big)) == 2
    assert call_scan_grouped(lib, scan_args(**big), 1) == 2
    assert lib.ssm_scan_workspace_bytes(1, 1 << 30, 1 << 40, 16, 1) == -1
    assert lib.ssm_scan_workspace_bytes_grouped(1, 1 << 30, 1 << 40, 16, 1, 1) == -1
    assert lib.ssm_scan_bwd_workspace_bytes(1, 1 << 30, 1 << 40, 16, 1) == -1
    assert call_conv(lib, batch=1, seqlen=1 << 40, dim=1 << 30) == 2
    assert call_upd(lib, upd_args(batch=1 << 62, dim=4)) == 2
    a = dict(state=P + 192 * MB, x=P, w=P + 64 * MB, bias=P + 128 * MB, out=P + 256 * MB)
    assert lib.ssm_conv1d_update(a["state"], a["x"], a["w"], a["bias"], 1, a["out"], 1 << 62, 4, 4, 1, None) == 2


def _noalloc_call(lib, **kw):
    """ssm_scan_fwd_noalloc on fake, non-overlapping addresses (never dereferenced:
    every case here is refused on the host)."""
    G = 1 << 30
    a = dict(u=P, delta=P + G, A=P + 2 * G, B=P + 3 * G, C=P + 4 * G, D=None, z=None, delta_bias=None,
             out=P + 5 * G, last=None, batch=4, dim=64, seqlen=131072, dstate=16, dtype=_lib.SSM_BF16)
    a.update(kw)
    return lib.ssm_scan_fwd_noalloc(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["delta_bias"], 1,
                                    a["out"], a["last"], a["batch"], a["dim"], a["seqlen"], a["dstate"], a["dtype"],
                                    None)


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    """A valid call whose workspace exceeds the fixed array is SSM_ERR_SCRATCH,
    decided on the host before the device is touched."""
    cap = lib.ssm_scan_noalloc_max_workspace_bytes()
    assert cap == 32 << 20
    # batch 4 x 131072 steps x N 16: 4 * 131072 * 128 bytes of staged B/C > 32 MiB
    assert lib.ssm_scan_workspace_bytes(4, 64, 131072, 16, _lib.SSM_BF16) > cap
    code = _noalloc_call(lib)
    assert code == 9 and _lib.status_string(code).startswith("SSM_ERR_SCRATCH")


@pytest.mark.parametrize("kw,code", [(dict(u=None), 1), (dict(out=P + 1), 3), (dict(out=P + 64), 6),
                                     (dict(dtype=7), 5), (dict(dstate=5), 4), (dict(batch=0), 2)],
                         ids=["null", "misaligned", "alias", "dtype", "dstate", "shape"])
def test_noalloc_checks_arguments_before_its_scratch(lib, kw, code):
    """Over-large sizes with a bad argument get the scan's own code for that
    argument, not SSM_ERR_SCRATCH: the argument checks come first."""
    assert _noalloc_call(lib, **kw) == code


def test_force_scan_path_hook(lib):
    """The kernel-selection hook: known paths are accepted (restoring the
    default last), anything else is SSM_ERR_SHAPE; no device is touched."""
    for path in (1, 2, 3, 4, 0):
        assert lib.ssm_force_scan_path(path, -1) == 0
    assert lib.ssm_force_scan_path(4, 2) == 0
    assert lib.ssm_force_scan_path(5, -1) == 2
    assert lib.ssm_force_scan_path(-1, -1) == 2
    assert lib.ssm_force_scan_path(0, -1) == 0
