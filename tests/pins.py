"""Pins for the float64 oracle: checks against facts the oracle does not define.

Each ``pin_*`` takes a loaded oracle library (the real one, or a mutated copy
in ``test_oracle_mutations.py``) and raises AssertionError when the oracle
disagrees with an independent route to the same answer:

* brute force:   the unrolled closed-form sum over the input history, using
                 exp of the summed timesteps (not a product of per-step decays);
* time-invariant: with Delta, B, C constant in time the scan is a causal
                 convolution with kernel K_k = sum_n C_n exp(k Delta A_n) Delta B_n,
                 evaluated with numpy.convolve, and for a unit step input it has a
                 geometric-series closed form;
* associative:   a Hillis-Steele log-depth inclusive scan of (dA, dB u) pairs
                 (the "parallel scan for training, O(N log N)" of the
                 "Efficient Scan" section of the Mamba README);
* limits:        Delta -> 0 leaves y = D u silu(z);  A -> -inf makes the model
                 memoryless;
* invariances:   linear in u, causal, unchanged by B -> cB, C -> C/c, and
                 equivariant under a permutation of channels;
* decode:        chaining the single-token update over L tokens from a zero
                 state reproduces the full scan exactly;
* initial state: the unrolled sum with the initial state's decay term
                 exp(A_n sum_{r<=t} Delta_r) h0_n added, and a sequence cut
                 anywhere and scanned in two pieces (the second from the first's
                 final state) reproducing the whole scan exactly;
* causal conv:   the impulse response is the reversed taps; numpy.convolve of
                 the carried state followed by the input gives every output and
                 the final state; a split sequence and a chain of decode steps
                 reproduce the whole convolution exactly;
* groups:        with B and C per channel group, the unrolled sum reading each
                 channel's own group, the grouped decode chain, and finite
                 differences of the grouped gradients;
* backward from a state: finite differences of <dout, out> + <dlast,
                 last_state> for every input and the initial state, and a
                 sequence differentiated in two pieces equal to the whole;
* backward:      central finite differences of L = sum(dout * out) through the
                 forward oracle for every input; and L = <du, u> (out is
                 linear in u), L = <dB, B> = <dC, C> without the D skip (out
                 is then linear in B and in C).

Softplus and sigmoid are taken from numpy/scipy library routines here
(``np.logaddexp``, ``scipy.special.expit``), never from the oracle.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import expit

import oracle

REL = 1e-12


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def tiny_case(seed, bt=2, L=12, dim=3, N=4, random_a=True, softplus=True,
              with_z=True, with_d=True, with_bias=True, groups=None):
    r = _rng(seed)
    u = r.standard_normal((bt, L, dim))
    delta = r.standard_normal((bt, L, dim)) * 0.5
    z = r.standard_normal((bt, L, dim)) if with_z else None
    bc_shape = (bt, N, L) if groups is None else (bt, groups, N, L)
    B = r.standard_normal(bc_shape)
    C = r.standard_normal(bc_shape)
    if random_a:
        A = -np.exp(r.standard_normal((dim, N)))
    else:
        A = np.tile(-np.arange(1.0, N + 1), (dim, 1))
    D = r.standard_normal(dim) if with_d else None
    bias = r.uniform(-3.0, 0.5, dim) if with_bias else None
    if not softplus:
        delta = np.abs(delta) * 0.3   # keep the raw timestep positive and moderate
    return dict(u=u, delta=delta, A=A, B=B, C=C, D=D, z=z, delta_bias=bias, softplus=softplus)


def _timestep(case):
    x = case["delta"] + (0.0 if case["delta_bias"] is None else case["delta_bias"][None, None, :])
    return np.logaddexp(0.0, x) if case["softplus"] else x


def _gate(case):
    z = case["z"]
    return 1.0 if z is None else z * expit(z)


def _close(got, ref, rel=REL, what=""):
    scale = max(1.0, float(np.max(np.abs(ref))))
    err = float(np.max(np.abs(got - ref)))
    assert err <= rel * scale, f"{what}: max|err| {err:.3e} > {rel:.1e} * {scale:.3e}"


def brute_force(case, h0=None):
    """y_t = sum_n C[n,t] (exp(A_n sum_{r<=t} Delta_r) h0_n
    + sum_{s<=t} exp(A_n sum_{r=s+1..t} Delta_r) Delta_s B[n,s] u_s) + D u_t, times
    silu(z_t) (h0 = 0 unless given); also the state after the last step.  With
    grouped B, C of shape (batch, G, N, L), channel d takes block d // (dim // G)."""
    u, A, B, C = case["u"], case["A"], case["B"], case["C"]
    bt, L, dim = u.shape
    N = A.shape[1]
    per = dim // (1 if B.ndim == 3 else B.shape[1])
    dlt = _timestep(case)
    Dv = np.zeros(dim) if case["D"] is None else case["D"]
    y = np.zeros_like(u)
    last = np.zeros((bt, dim, N))
    for b in range(bt):
        for d in range(dim):
            Bd, Cd = (B[b], C[b]) if B.ndim == 3 else (B[b, d // per], C[b, d // per])
            for t in range(L):
                h = np.zeros(N)
                if h0 is not None:
                    h += np.exp(A[d] * float(np.sum(dlt[b, :t + 1, d]))) * h0[b, d]
                for s in range(t + 1):
                    span = float(np.sum(dlt[b, s + 1:t + 1, d]))
                    h += np.exp(A[d] * span) * dlt[b, s, d] * Bd[:, s] * u[b, s, d]
                y[b, t, d] = float(np.dot(Cd[:, t], h)) + Dv[d] * u[b, t, d]
                if t == L - 1:
                    last[b, d] = h
    return y * _gate(case), last


def run_oracle(case, lib, h0=None):
    return oracle.scan(case["u"], case["delta"], case["A"], case["B"], case["C"], case["D"],
                       case["z"], case["delta_bias"], case["softplus"], lib=lib, initial_state=h0)


# --------------------------------------------------------------------------- pins

def pin_brute_force(lib):
    for seed, kw in [(1, {}), (2, dict(softplus=False)), (3, dict(random_a=False, N=3)),
                     (4, dict(with_z=False, with_d=False, with_bias=False)), (5, dict(L=16, dim=2, N=2))]:
        case = tiny_case(seed, **kw)
        out, last = run_oracle(case, lib)
        ref, ref_last = brute_force(case)
        _close(out, ref, what=f"brute out seed {seed}")
        _close(last, ref_last, what=f"brute last_state seed {seed}")


def pin_time_invariant_convolution(lib):
    r = _rng(11)
    bt, L, dim, N = 2, 40, 3, 4
    A = -np.exp(r.standard_normal((dim, N)))
    raw = r.uniform(-2.0, 0.0, dim)                   # constant per channel
    delta = np.broadcast_to(raw[None, None, :], (bt, L, dim)).copy()
    beta = r.standard_normal((bt, N))
    gamma = r.standard_normal((bt, N))
    B = np.repeat(beta[:, :, None], L, axis=2)
    C = np.repeat(gamma[:, :, None], L, axis=2)
    D = r.standard_normal(dim)
    u = r.standard_normal((bt, L, dim))
    case = dict(u=u, delta=delta, A=A, B=B, C=C, D=D, z=None, delta_bias=None, softplus=True)
    out, _ = run_oracle(case, lib)
    dl = np.logaddexp(0.0, raw)                       # library softplus
    k = np.arange(L)
    for b in range(bt):
        for d in range(dim):
            K = (gamma[b][None, :] * np.exp(np.outer(k, dl[d] * A[d])) * dl[d] * beta[b][None, :]).sum(1)
            ref = np.convolve(u[b, :, d], K)[:L] + D[d] * u[b, :, d]
            _close(out[b, :, d], ref, what=f"LTI conv b{b} d{d}")
    # unit step input: y_t = D + sum_n C_n Delta B_n (1 - e^{(t+1) Delta A_n}) / (1 - e^{Delta A_n})
    case["u"] = np.ones((bt, L, dim))
    out, last = run_oracle(case, lib)
    for b in range(bt):
        for d in range(dim):
            q = np.exp(dl[d] * A[d])
            geo = (1.0 - np.exp(np.outer(k + 1, dl[d] * A[d]))) / (1.0 - q)[None, :]
            ref = (gamma[b] * dl[d] * beta[b] * geo).sum(1) + D[d]
            _close(out[b, :, d], ref, what=f"LTI step b{b} d{d}")
            _close(last[b, d], dl[d] * beta[b] * geo[-1], what=f"LTI step state b{b} d{d}")


def hillis_steele_states(a, bb):
    """Inclusive log-depth scan of x_t = a_t x_{t-1} + b_t over axis 0 (x_{-1} = 0)."""
    a = a.copy()
    bb = bb.copy()
    L = a.shape[0]
    off = 1
    while off < L:
        a_new, b_new = a.copy(), bb.copy()
        a_new[off:] = a[off:] * a[:-off]
        b_new[off:] = a[off:] * bb[:-off] + bb[off:]
        a, bb = a_new, b_new
        off *= 2
    return bb


def pin_associative_scan(lib):
    for seed in (21, 22):
        case = tiny_case(seed, bt=2, L=16, dim=3, N=4)
        out, last = run_oracle(case, lib)
        dlt = _timestep(case)
        u, A, B, C = case["u"], case["A"], case["B"], case["C"]
        ref = np.zeros_like(u)
        for b in range(u.shape[0]):
            for d in range(u.shape[2]):
                a = np.exp(dlt[b, :, d][:, None] * A[d][None, :])
                bb = (dlt[b, :, d] * u[b, :, d])[:, None] * B[b].T
                h = hillis_steele_states(a, bb)
                ref[b, :, d] = (C[b].T * h).sum(1) + case["D"][d] * u[b, :, d]
                _close(last[b, d], h[-1], what="assoc last_state")
        _close(out, ref * _gate(case), what=f"assoc scan seed {seed}")


def pin_delta_to_zero(lib):
    case = tiny_case(31, L=10)
    case["delta_bias"] = np.full(case["u"].shape[2], -1e4)   # softplus(-1e4 + x) underflows to 0
    out, last = run_oracle(case, lib)
    ref = case["D"][None, None, :] * case["u"] * _gate(case)
    _close(out, ref, rel=1e-15, what="Delta->0 skip+gate")
    assert np.all(last == 0.0), "Delta->0 must leave the state at zero"


def pin_memoryless_limit(lib):
    case = tiny_case(32, L=10, softplus=False)
    case["delta"] = 0.1 + np.abs(case["delta"])              # Delta >= 0.1
    case["A"] = np.full_like(case["A"], -1e4)                # dA = exp(-1e3..) = 0
    case["delta_bias"] = None
    out, last = run_oracle(case, lib)
    u, B, C, dl = case["u"], case["B"], case["C"], case["delta"]
    cb = np.einsum("bnt,bnt->bt", C, B)                      # sum_n C_n B_n per (b, t)
    ref = (dl * u * cb[:, :, None] + case["D"][None, None, :] * u) * _gate(case)
    _close(out, ref, what="A->-inf memoryless")
    ref_last = (dl[:, -1, :] * u[:, -1, :])[:, :, None] * B[:, :, -1][:, None, :]
    _close(last, ref_last, what="A->-inf state")


def pin_linear_in_u(lib):
    c1 = tiny_case(41, L=14)
    c2 = dict(c1)
    c2["u"] = _rng(42).standard_normal(c1["u"].shape)
    c3 = dict(c1)
    c3["u"] = 2.5 * c1["u"] - 0.75 * c2["u"]
    o1, s1 = run_oracle(c1, lib)
    o2, s2 = run_oracle(c2, lib)
    o3, s3 = run_oracle(c3, lib)
    _close(o3, 2.5 * o1 - 0.75 * o2, what="linearity out")
    _close(s3, 2.5 * s1 - 0.75 * s2, what="linearity state")


def pin_causal(lib):
    c1 = tiny_case(51, L=14)
    o1, _ = run_oracle(c1, lib)
    t0 = 6
    c2 = dict(c1)
    c2["u"] = c1["u"].copy()
    c2["u"][:, t0, :] += 1.0
    o2, _ = run_oracle(c2, lib)
    assert np.array_equal(o1[:, :t0], o2[:, :t0]), "output before t0 changed: not causal"
    assert np.all(np.abs(o1[:, t0:] - o2[:, t0:]).max(axis=1) > 0), "perturbation at t0 had no effect"


def pin_bc_scale(lib):
    c1 = tiny_case(61, L=14)
    c2 = dict(c1)
    c2["B"] = c1["B"] * 3.0
    c2["C"] = c1["C"] / 3.0
    o1, s1 = run_oracle(c1, lib)
    o2, s2 = run_oracle(c2, lib)
    _close(o2, o1, what="B->cB, C->C/c")
    _close(s2, 3.0 * s1, what="state scales with B")


def pin_channel_permutation(lib):
    c1 = tiny_case(71, L=9, dim=5, N=3)
    perm = np.array([3, 0, 4, 1, 2])
    c2 = dict(c1)
    for k in ("u", "delta", "z"):
        c2[k] = c1[k][:, :, perm]
    c2["A"] = c1["A"][perm]
    c2["D"] = c1["D"][perm]
    c2["delta_bias"] = c1["delta_bias"][perm]
    o1, s1 = run_oracle(c1, lib)
    o2, s2 = run_oracle(c2, lib)
    assert np.array_equal(o2, o1[:, :, perm]), "channel permutation changed the arithmetic"
    assert np.array_equal(s2, s1[:, perm]), "channel permutation changed the state"


def pin_decode_chain_equals_scan(lib):
    for kw in ({}, dict(softplus=False), dict(with_z=False, with_bias=False)):
        case = tiny_case(81, bt=3, L=11, dim=4, N=4, **kw)
        out, last = run_oracle(case, lib)
        bt, L, dim = case["u"].shape
        N = case["A"].shape[1]
        state = np.zeros((bt, dim, N))
        for t in range(L):
            o = oracle.step(state, case["u"][:, t, :], case["delta"][:, t, :], case["A"],
                            np.ascontiguousarray(case["B"][:, :, t]), np.ascontiguousarray(case["C"][:, :, t]),
                            case["D"], None if case["z"] is None else case["z"][:, t, :],
                            case["delta_bias"], case["softplus"], lib=lib)
            assert np.array_equal(o, out[:, t, :]), f"decode step {t} differs from scan"
        assert np.array_equal(state, last), "decode chain final state differs from scan"


def pin_initial_state_brute_force(lib):
    for seed, kw in [(91, {}), (92, dict(softplus=False, with_z=False)), (93, dict(random_a=False, N=3))]:
        case = tiny_case(seed, **kw)
        bt, L, dim = case["u"].shape
        h0 = _rng(seed + 100).standard_normal((bt, dim, case["A"].shape[1]))
        out, last = run_oracle(case, lib, h0)
        ref, ref_last = brute_force(case, h0)
        _close(out, ref, what=f"initial-state brute out seed {seed}")
        _close(last, ref_last, what=f"initial-state brute last_state seed {seed}")


def _cut(case, lo, hi):
    c = dict(case)
    for k in ("u", "delta", "z"):
        if case[k] is not None:
            c[k] = np.ascontiguousarray(case[k][:, lo:hi])
    for k in ("B", "C"):
        c[k] = np.ascontiguousarray(case[k][..., lo:hi])
    return c


def pin_split_equals_whole(lib):
    for seed, cut in [(95, 1), (96, 7), (97, 11)]:
        case = tiny_case(seed, bt=2, L=12, dim=3, N=4)
        out, last = run_oracle(case, lib)
        o1, s1 = run_oracle(_cut(case, 0, cut), lib)
        o2, s2 = run_oracle(_cut(case, cut, 12), lib, s1)
        assert np.array_equal(np.concatenate([o1, o2], axis=1), out), f"split at {cut} changed the output"
        assert np.array_equal(s2, last), f"split at {cut} changed the final state"


def conv_case(seed, bt=2, L=10, dim=3, W=4, with_bias=True, with_state=True):
    r = _rng(seed)
    return dict(x=r.standard_normal((bt, L, dim)), w=r.standard_normal((dim, W)),
                bias=r.standard_normal(dim) if with_bias else None,
                state=r.standard_normal((bt, dim, W - 1)) if with_state else None)


def pin_conv_impulse(lib):
    for W in (2, 3, 4):
        c = conv_case(120 + W, bt=1, L=12, dim=2, W=W, with_bias=False, with_state=False)
        x = np.zeros((1, 12, 2))
        x[0, 5, 1] = 1.0
        out, _ = oracle.conv1d(x, c["w"], None, False, None, lib=lib)
        want = np.zeros((12,))
        want[5:5 + W] = c["w"][1, ::-1]
        assert np.array_equal(out[0, :, 1], want), f"impulse response, width {W}"
        assert np.array_equal(out[0, :, 0], np.zeros(12)), "impulse leaked into another channel"


def pin_conv_numpy(lib):
    for seed, kw in [(130, {}), (131, dict(with_state=False)), (132, dict(W=2, with_bias=False)),
                     (133, dict(L=2, W=4)), (134, dict(L=1, W=3))]:
        c = conv_case(seed, **kw)
        for silu in (False, True):
            out, st = oracle.conv1d(c["x"], c["w"], c["bias"], silu, c["state"], lib=lib)
            bt, L, dim = c["x"].shape
            W = c["w"].shape[1]
            for b in range(bt):
                for d in range(dim):
                    prev = np.zeros(W - 1) if c["state"] is None else c["state"][b, d]
                    seq = np.concatenate([prev, c["x"][b, :, d]])
                    y = np.convolve(seq, c["w"][d, ::-1], mode="valid")
                    y = y + (0.0 if c["bias"] is None else c["bias"][d])
                    if silu:
                        y = y * expit(y)
                    _close(out[b, :, d], y, what=f"conv seed {seed} ({b},{d})")
                    assert np.array_equal(st[b, d], seq[len(seq) - (W - 1):]), f"conv state seed {seed}"


def pin_conv_split_and_decode(lib):
    c = conv_case(140, bt=2, L=11, dim=3, W=4)
    out, st = oracle.conv1d(c["x"], c["w"], c["bias"], True, c["state"], lib=lib)
    for cut in (1, 2, 7):
        o1, s1 = oracle.conv1d(np.ascontiguousarray(c["x"][:, :cut]), c["w"], c["bias"], True, c["state"], lib=lib)
        o2, s2 = oracle.conv1d(np.ascontiguousarray(c["x"][:, cut:]), c["w"], c["bias"], True, s1, lib=lib)
        assert np.array_equal(np.concatenate([o1, o2], axis=1), out), f"conv split at {cut}"
        assert np.array_equal(s2, st), f"conv split state at {cut}"
    state = c["state"].copy()
    for t in range(11):
        o = oracle.conv1d_update(state, np.ascontiguousarray(c["x"][:, t]), c["w"], c["bias"], True, lib=lib)
        assert np.array_equal(o, out[:, t]), f"conv decode step {t}"
    assert np.array_equal(state, st), "conv decode final state"


def _loss(case, dout, lib):
    out, _ = run_oracle(case, lib)
    return float(np.sum(dout * out))


def _grads(case, dout, lib):
    return oracle.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], case["D"], case["z"],
                           case["delta_bias"], case["softplus"], dout, lib=lib)


GRAD_OF = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "z": "dz",
           "delta_bias": "ddelta_bias"}


def pin_bwd_finite_differences(lib):
    for seed, kw in [(201, {}), (202, dict(softplus=False)), (203, dict(with_z=False, with_d=False, with_bias=False)),
                     (204, dict(random_a=False, N=2))]:
        case = tiny_case(seed, bt=2, L=6, dim=2, N=kw.pop("N", 3), **kw)
        dout = _rng(seed + 50).standard_normal(case["u"].shape)
        g = _grads(case, dout, lib)
        for name, gname in GRAD_OF.items():
            if case[name] is None:
                continue
            base = case[name]
            fd = np.zeros_like(base)
            for idx in np.ndindex(base.shape):
                eps = 1e-6 * max(1.0, abs(float(base[idx])))
                for sgn in (1.0, -1.0):
                    c = dict(case)
                    c[name] = base.copy()
                    c[name][idx] += sgn * eps
                    fd[idx] += sgn * _loss(c, dout, lib) / (2.0 * eps)
            scale = max(1.0, float(np.max(np.abs(fd))))
            err = float(np.max(np.abs(g[gname] - fd)))
            assert err <= 2e-6 * scale, f"d{name} seed {seed}: |analytic - finite difference| {err:.2e}"


def pin_bwd_homogeneity(lib):
    for seed in (211, 212):
        case = tiny_case(seed, bt=2, L=9, dim=3, N=4)
        dout = _rng(seed + 1).standard_normal(case["u"].shape)
        lval = _loss(case, dout, lib)
        g = _grads(case, dout, lib)
        _close(np.array([np.sum(g["du"] * case["u"])]), np.array([lval]), what="<du, u> = L")
        case = tiny_case(seed, bt=2, L=9, dim=3, N=4, with_d=False)
        lval = _loss(case, dout, lib)
        g = _grads(case, dout, lib)
        _close(np.array([np.sum(g["dB"] * case["B"])]), np.array([lval]), what="<dB, B> = L")
        _close(np.array([np.sum(g["dC"] * case["C"])]), np.array([lval]), what="<dC, C> = L")


def pin_grouped_brute_force(lib):
    """B and C per channel group: the unrolled sum with each channel reading
    its own group's B and C; with ngroups = dim every channel has its own."""
    for seed, kw in [(301, dict(dim=4, groups=2)), (302, dict(dim=6, groups=3, softplus=False)),
                     (303, dict(dim=3, groups=3, N=2)), (304, dict(dim=4, groups=1))]:
        case = tiny_case(seed, L=9, **kw)
        bt, _, dim = case["u"].shape
        h0 = _rng(seed + 7).standard_normal((bt, dim, case["A"].shape[1]))
        for init in (None, h0):
            out, last = run_oracle(case, lib, init)
            ref, ref_last = brute_force(case, init)
            _close(out, ref, what=f"grouped brute out seed {seed}")
            _close(last, ref_last, what=f"grouped brute last_state seed {seed}")


def pin_grouped_decode_chain(lib):
    """The grouped decode step chained over L tokens reproduces the grouped scan
    exactly, and one decode step from a random state equals the one-step
    unrolled sum (decay of the state plus the new input's term)."""
    case = tiny_case(311, bt=2, L=8, dim=6, N=3, groups=3)
    bt, L, dim = case["u"].shape
    N = case["A"].shape[1]
    out, last = run_oracle(case, lib)
    state = np.zeros((bt, dim, N))
    for t in range(L):
        o = oracle.step(state, case["u"][:, t, :], case["delta"][:, t, :], case["A"],
                        np.ascontiguousarray(case["B"][:, :, :, t]), np.ascontiguousarray(case["C"][:, :, :, t]),
                        case["D"], case["z"][:, t, :], case["delta_bias"], case["softplus"], lib=lib)
        assert np.array_equal(o, out[:, t, :]), f"grouped decode step {t} differs from the grouped scan"
    assert np.array_equal(state, last), "grouped decode chain final state differs from the grouped scan"
    one = _cut(case, 0, 1)
    h0 = _rng(312).standard_normal((bt, dim, N))
    ref, ref_last = brute_force(one, h0)
    st = h0.copy()
    o = oracle.step(st, one["u"][:, 0, :], one["delta"][:, 0, :], one["A"], np.ascontiguousarray(one["B"][..., 0]),
                    np.ascontiguousarray(one["C"][..., 0]), one["D"], one["z"][:, 0, :], one["delta_bias"],
                    one["softplus"], lib=lib)
    _close(o, ref[:, 0, :], what="grouped decode step vs brute force")
    _close(st, ref_last, what="grouped decode state vs brute force")


def pin_grouped_bwd_finite_differences(lib):
    """Grouped gradients: dB and dC sum over the channels of each group only."""
    case = tiny_case(321, bt=2, L=5, dim=4, N=2, groups=2)
    dout = _rng(322).standard_normal(case["u"].shape)
    g = _grads(case, dout, lib)
    assert g["dB"].shape == case["B"].shape and g["dC"].shape == case["C"].shape
    for name, gname in GRAD_OF.items():
        base = case[name]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            eps = 1e-6 * max(1.0, abs(float(base[idx])))
            for sgn in (1.0, -1.0):
                c = dict(case)
                c[name] = base.copy()
                c[name][idx] += sgn * eps
                fd[idx] += sgn * _loss(c, dout, lib) / (2.0 * eps)
        scale = max(1.0, float(np.max(np.abs(fd))))
        err = float(np.max(np.abs(g[gname] - fd)))
        assert err <= 2e-6 * scale, f"grouped d{name}: |analytic - finite difference| {err:.2e}"


def _grads_from(case, dout, h0, dlast, lib):
    return oracle.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], case["D"], case["z"],
                           case["delta_bias"], case["softplus"], dout, lib=lib, initial_state=h0, dlast=dlast)


def pin_bwd_from_state_finite_differences(lib):
    """Backward of the scan from a given state, with the final state in the
    loss: central finite differences of L = <dout, out> + <dlast, last_state>
    for every input and for the initial state (dinitial_state)."""
    # (without softplus and bias, Delta = 0.3 |delta_raw| >= 0 keeps the recurrence bounded)
    for seed, kw in [(331, dict(dim=2)),
                     (332, dict(dim=4, groups=2, with_z=False, softplus=False, with_bias=False))]:
        case = tiny_case(seed, bt=2, L=6, N=3, **kw)
        bt, L, dim = case["u"].shape
        N = case["A"].shape[1]
        r = _rng(seed + 1)
        h0 = r.standard_normal((bt, dim, N))
        dlast = r.standard_normal((bt, dim, N))
        dout = r.standard_normal(case["u"].shape)

        def loss(c, h):
            out, last = run_oracle(c, lib, h)
            return float(np.sum(dout * out) + np.sum(dlast * last))

        g = _grads_from(case, dout, h0, dlast, lib)
        for name, gname in list(GRAD_OF.items()) + [("initial_state", "dinitial_state")]:
            base = h0 if name == "initial_state" else case[name]
            if base is None:
                continue
            fd = np.zeros_like(base)
            for idx in np.ndindex(base.shape):
                eps = 1e-6 * max(1.0, abs(float(base[idx])))
                for sgn in (1.0, -1.0):
                    pert = base.copy()
                    pert[idx] += sgn * eps
                    c, h = (case, pert) if name == "initial_state" else (dict(case, **{name: pert}), h0)
                    fd[idx] += sgn * loss(c, h) / (2.0 * eps)
            scale = max(1.0, float(np.max(np.abs(fd))))
            err = float(np.max(np.abs(g[gname] - fd)))
            assert err <= 2e-6 * scale, f"from-state d{name} seed {seed}: |analytic - finite difference| {err:.2e}"


def pin_bwd_split_equals_whole(lib):
    """A sequence cut in two and differentiated piece by piece -- the second
    piece from the first piece's final state, the first piece taking the
    second piece's dinitial_state as its dlast -- gives the whole backward."""
    for seed, cut in [(341, 1), (342, 5), (343, 9)]:
        case = tiny_case(seed, bt=2, L=10, dim=3, N=4)
        bt, L, dim = case["u"].shape
        r = _rng(seed + 7)
        h0 = r.standard_normal((bt, dim, 4))
        dlast = r.standard_normal((bt, dim, 4))
        dout = r.standard_normal(case["u"].shape)
        whole = _grads_from(case, dout, h0, dlast, lib)
        c1, c2 = _cut(case, 0, cut), _cut(case, cut, L)
        _, hmid = run_oracle(c1, lib, h0)
        g2 = _grads_from(c2, np.ascontiguousarray(dout[:, cut:]), hmid, dlast, lib)
        g1 = _grads_from(c1, np.ascontiguousarray(dout[:, :cut]), h0, g2["dinitial_state"], lib)
        for k in ("du", "ddelta", "dz"):
            _close(np.concatenate([g1[k], g2[k]], axis=1), whole[k], what=f"split backward {k}, cut {cut}")
        for k in ("dB", "dC"):
            _close(np.concatenate([g1[k], g2[k]], axis=-1), whole[k], what=f"split backward {k}, cut {cut}")
        for k in ("dA", "dD", "ddelta_bias"):
            _close(g1[k] + g2[k], whole[k], what=f"split backward {k}, cut {cut}")
        _close(g1["dinitial_state"], whole["dinitial_state"], what=f"split backward dinitial, cut {cut}")


def pin_scalar_functions(lib):
    sp = lambda x: oracle.softplus(x, lib=lib)
    si = lambda x: oracle.silu(x, lib=lib)
    assert abs(sp(0.0) - math.log(2.0)) <= 1e-16
    assert abs(sp(math.log(math.e - 1.0)) - 1.0) <= 4e-16
    for x in (-745.0, -300.0, -40.0, -1e-3, 0.3, 3.0, 35.0, 700.0):
        assert abs(sp(x) - sp(-x) - x) <= 4e-16 * max(1.0, abs(x)), f"softplus odd-part identity at {x}"
        ref = float(np.logaddexp(0.0, x))
        assert abs(sp(x) - ref) <= 2e-16 * max(ref, 1e-300) + 1e-320, f"softplus({x})"
    for x in (-30.0, -2.0, -0.5, 0.0, 0.7, 4.0, 25.0):
        assert abs(si(x) - si(-x) - x) <= 4e-16 * max(1.0, abs(x)), f"silu odd-part identity at {x}"
        ref = x * float(expit(x))
        assert abs(si(x) - ref) <= 4e-16 * max(abs(ref), 1e-300), f"silu({x})"
    assert si(math.log(3.0)) - 0.75 * math.log(3.0) < 4e-16


ALL_PINS = [pin_brute_force, pin_time_invariant_convolution, pin_associative_scan,
            pin_delta_to_zero, pin_memoryless_limit, pin_linear_in_u, pin_causal,
            pin_bc_scale, pin_channel_permutation, pin_decode_chain_equals_scan,
            pin_initial_state_brute_force, pin_split_equals_whole, pin_conv_impulse, pin_conv_numpy,
            pin_conv_split_and_decode, pin_bwd_finite_differences, pin_bwd_homogeneity,
            pin_grouped_brute_force, pin_grouped_decode_chain, pin_grouped_bwd_finite_differences,
            pin_bwd_from_state_finite_differences, pin_bwd_split_equals_whole, pin_scalar_functions]
