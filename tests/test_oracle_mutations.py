"""Planted mistakes in the oracle must each fail at least one pin.

Each mutation rewrites one line of a copy of ``oracle/kda_oracle.c`` (a
dropped term, a wrong sign, index or operand), builds the copy with gcc on the
CPU and runs every pin of ``oracle_pins`` against it.  A mutation that no pin
notices means the pins leave that part of the oracle unchecked.
"""

from __future__ import annotations

import pytest

from oracle import kda_oracle as ko

import oracle_pins as pins

MUTATIONS = [
    # a3 update
    ("decay dropped", "M[i * dv + j] = at[i] * S[i * dv + j];", "M[i * dv + j] = S[i * dv + j];"),
    ("decay on the value index", "M[i * dv + j] = at[i] * S[i * dv + j];", "M[i * dv + j] = at[j % dk] * S[i * dv + j];"),
    ("write sign flipped", "S[i * dv + j] = M[i * dv + j] + bt * kt[i] * (vt[j] - u[j]);",
     "S[i * dv + j] = M[i * dv + j] - bt * kt[i] * (vt[j] - u[j]);"),
    ("erase term sign", "S[i * dv + j] = M[i * dv + j] + bt * kt[i] * (vt[j] - u[j]);",
     "S[i * dv + j] = M[i * dv + j] + bt * kt[i] * (vt[j] + u[j]);"),
    ("beta dropped", "S[i * dv + j] = M[i * dv + j] + bt * kt[i] * (vt[j] - u[j]);",
     "S[i * dv + j] = M[i * dv + j] + kt[i] * (vt[j] - u[j]);"),
    ("prediction from the undecayed state", "acc += kt[i] * M[i * dv + j];", "acc += kt[i] * S[i * dv + j];"),
    ("prediction with q", "acc += kt[i] * M[i * dv + j];", "acc += qt[i] * M[i * dv + j];"),
    # a4 readout
    ("readout before the update", "            for (int i = 0; i < dk; ++i)\n                acc += qt[i] * S[i * dv + j];\n            o[t * os + j] = acc;",
     "            for (int i = 0; i < dk; ++i)\n                acc += qt[i] * M[i * dv + j];\n            o[t * os + j] = acc;"),
    ("readout transposed", "            for (int i = 0; i < dk; ++i)\n                acc += qt[i] * S[i * dv + j];\n            o[t * os + j] = acc;",
     "            for (int i = 0; i < dk; ++i)\n                acc += qt[i] * S[j * dk + i];\n            o[t * os + j] = acc;"),
    # a1 conv
    ("tap order reversed", "acc += w[j] * tail[j * ts];", "acc += w[W - 2 - j] * tail[j * ts];"),
    ("current-token tap on tap 0", "acc += w[W - 1] * x[t * xs];", "acc += w[0] * x[t * xs];"),
    ("no SiLU", "y[t * ys] = silu(acc);", "y[t * ys] = acc;"),
    ("tail not advanced", "tail[(W - 2) * ts] = x[t * xs];", "tail[(W - 2) * ts] = tail[(W - 2) * ts];"),
    # a2 L2
    ("eps outside the root", "double r = 1.0 / sqrt(ss + eps);", "double r = 1.0 / (sqrt(ss) + eps);"),
    ("q not normalised", "l2norm(dk, qc + t * dk, eps_l2);", ";"),
    ("k not normalised", "l2norm(dk, kc + t * dk, eps_l2);", ";"),
    # a5 gated norm
    ("sum instead of mean", "ms = ms / dv;", "ms = ms;"),
    ("gate dropped", "y[j] = wn[j] * (o[j] * r) * sigmoid(g[j]);", "y[j] = wn[j] * (o[j] * r);"),
    ("norm weight dropped", "y[j] = wn[j] * (o[j] * r) * sigmoid(g[j]);", "y[j] = (o[j] * r) * sigmoid(g[j]);"),
    ("gate as a value", "y[j] = wn[j] * (o[j] * r) * sigmoid(g[j]);", "y[j] = wn[j] * (o[j] * r) * g[j];"),
    # layer indexing
    ("beta of head 0 for every head", "const double *be = beta + (long)t0 * H + h;", "const double *be = beta + (long)t0 * H;"),
    ("alpha of head 0 for every head", "const double *al = alpha + (long)t0 * H * dk + (long)h * dk;",
     "const double *al = alpha + (long)t0 * H * dk;"),
    # chunked form
    ("chunk: beta dropped from W", "acc += T[r * C + s] * bc[s * bs] * exp(G[s * dk + i]) *",
     "acc += T[r * C + s] * exp(G[s * dk + i]) *"),
    ("chunk: diagonal dropped from P", "for (int s = 0; s <= r; ++s) {", "for (int s = 0; s < r; ++s) {"),
    ("chunk: wrong carry decay", "acc += exp(G[(n - 1) * dk + i] - G[s * dk + i]) *", "acc += exp(-G[s * dk + i]) *"),
    ("chunk: A scaled by beta_s", "A[r * C + s] = bc[r * bs] * acc;", "A[r * C + s] = bc[s * bs] * acc;"),
    ("chunk: T sign", "acc -= A[r * C + s] * T[s * C + c];", "acc += A[r * C + s] * T[s * C + c];"),
]


@pytest.fixture(scope="module")
def source():
    return ko.SRC.read_text()


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new, source, tmp_path):
    assert source.count(old) == 1, f"mutation site for '{name}' is not unique"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib = ko.compile_source(src, tmp_path / "libmutant.so")
    o = ko.Oracle(lib)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, RuntimeError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake '{name}'"
