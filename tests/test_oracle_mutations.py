"""Plant plausible mistakes in copies of the oracle and check the pins catch them.

Each mutation is a textual edit of oracle.c compiled into a temporary library;
the real oracle is never modified.  A mutation that no pin rejects would mean
the pins leave part of the oracle unchecked.
"""
import os

import pytest

import oracle
import pins

MUTATIONS = [
    ("state update sign", "h[n] = dA * h[n] + dBu;", "h[n] = dA * h[n] - dBu;"),
    ("decay sign", "double dA = exp(dlt * Arow[n]);", "double dA = exp(-dlt * Arow[n]);"),
    ("dropped decay", "h[n] = dA * h[n] + dBu;", "h[n] = h[n] + dBu;"),
    ("dropped Delta in dB", "double dBu = (dlt * Bv[n * bc_stride]) * uv;",
     "double dBu = Bv[n * bc_stride] * uv;"),
    ("B/C transposed in readout", "y += Cv[n * bc_stride] * h[n];", "y += Bv[n * bc_stride] * h[n];"),
    ("dropped D skip", "y += Dd * uv;", ""),
    ("gate is z not silu(z)", "if (zp) y *= silu(*zp);", "if (zp) y *= *zp;"),
    ("readout uses h_{t-1}",
     "        h[n] = dA * h[n] + dBu;\n        y += Cv[n * bc_stride] * h[n];",
     "        y += Cv[n * bc_stride] * h[n];\n        h[n] = dA * h[n] + dBu;"),
    ("softplus without log1p", "log1p(exp(-fabs(x)))", "log(exp(-fabs(x)))"),
    ("softplus drops max", "(x > 0.0 ? x : 0.0) + ", ""),
    ("bias ignored", "delta_raw + (delta_bias ? delta_bias[d] : 0.0)", "delta_raw"),
    ("A indexed transposed", "A + d * N, (int)N, Bb + t", "A + d, (int)N, Bb + t"),
    ("B/C time index off by one", "Bb + t, Cb + t, L,", "Bb + (t ? t - 1 : 0), Cb + (t ? t - 1 : 0), L,"),
    ("silu sign", "return zv / (1.0 + exp(-zv));", "return zv / (1.0 + exp(zv));"),
    ("state written transposed", "last_state[(b * Dm + d) * N + n] = h[n];",
     "last_state[(b * N + n) * Dm + d] = h[n];"),
    ("decode ignores dt bias", "timestep(dt[i], dt_bias, (int)d, dt_softplus)",
     "timestep(dt[i], NULL, (int)d, dt_softplus)"),
    ("initial state ignored", "h[n] = initial_state ? initial_state[(b * Dm + d) * N + n] : 0.0;",
     "h[n] = 0.0;"),
    ("conv taps reversed", "acc += w[d * W + k] * conv_input(", "acc += w[d * W + (W - 1 - k)] * conv_input("),
    ("conv state oldest-last", "state_in[(b * Dm + d) * (W - 1) + (W - 1) + s]", "state_in[(b * Dm + d) * (W - 1) - 1 - s]"),
    ("conv without bias", "double acc = bias ? bias[d] : 0.0;\n            for (int k = 0; k < W; ++k)",
     "double acc = 0.0;\n            for (int k = 0; k < W; ++k)"),
    ("conv decode shifts the wrong way", "for (int k = 0; k + 1 < W - 1; ++k) st[k] = st[k + 1];",
     "for (int k = W - 2; k > 0; --k) st[k] = st[k - 1];"),
    ("adjoint without decay", "lam[n] = Cb[n * L + t] * dy + anext[n] * lam[n];", "lam[n] = Cb[n * L + t] * dy + lam[n];"),
    ("dA uses h_t", "dA[d * N + n] += lam[n] * dlt * a * hprev;", "dA[d * N + n] += lam[n] * dlt * a * h;"),
    ("dDelta drops B u", "ddl += lam[n] * (Ar[n] * a * hprev + Bb[n * L + t] * u[i]);", "ddl += lam[n] * (Ar[n] * a * hprev);"),
    ("softplus derivative sign", "ddl * sigmoid(xr)", "ddl * sigmoid(-xr)"),
    ("dB without Delta", "dB[(blk * N + n) * L + t] += lam[n] * dlt * u[i];",
     "dB[(blk * N + n) * L + t] += lam[n] * u[i];"),
    ("initial state read transposed", "h[n] = initial_state ? initial_state[(b * Dm + d) * N + n] : 0.0;",
     "h[n] = initial_state ? initial_state[(b * N + n) * Dm + d] : 0.0;"),
    ("group taken as channel remainder", "return b * ngroups + d / (dim / ngroups);",
     "return b * ngroups + d % ngroups;"),
    ("group batch stride dropped", "return b * ngroups + d / (dim / ngroups);", "return b + d / (dim / ngroups);"),
    ("decode ignores groups", "B + blk * N, C + blk * N, 1,", "B + b * N, C + b * N, 1,"),
    ("grouped dC summed into the batch row", "dC[(blk * N + n) * L + t] += dy * h;",
     "dC[(b * N + n) * L + t] += dy * h;"),
    ("backward ignores the initial state", "hs[n] = initial_state ? initial_state[sbase + n] : 0.0;",
     "hs[n] = 0.0;"),
    ("final-state adjoint ignored", "lam[n] = dlast ? dlast[sbase + n] : 0.0;", "lam[n] = 0.0;"),
    ("initial-state adjoint without the first decay", "dinitial[sbase + n] = anext[n] * lam[n];",
     "dinitial[sbase + n] = lam[n];"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new, tmp_path):
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {name}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "liboracle_mut.so")
    oracle.build(src=str(mutated), out=so)
    lib = oracle.load(so)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin rejects the mutation '{name}'"
