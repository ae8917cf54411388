"""Planted mistakes in the fp64 oracle are caught by its pins.

Each case takes a copy of an oracle source with one plausible slip (a dropped
term, a wrong sign, a wrong operand or mask, a missing factor):

* ``oracle/kda_oracle.c`` (the recurrence every parity test compares against),
  compiled and run against the independent torch float64 autograd of the
  literal recurrence (the pin of ``test_oracle_pins.py``);
* ``oracle/chunked.py`` (the chunked form behind the per-stage GPU checks),
  loaded and run against the recurrence (the chunked-equals-recurrent pin).

Every mutant must miss its pin by far more than the pin's 1e-12 tolerance; the
unmodified sources, taken the same way, must meet it. (Slips that change nothing, such
as an Akk diagonal that the unit-diagonal solve and the strictly lower dAkk mask
both ignore, are not listed.) This shows that the pins
would notice such a mistake in the oracle, not only that the oracle agrees
with them.
"""
import ctypes
import importlib.util
import os
import subprocess

import numpy as np
import pytest

import kda_inputs
import oracle
from tests.test_oracle_pins import _f64_inputs, _torch_literal

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, original text, mutated text): each original occurs exactly once in the source
MUTANTS = [
    # forward
    ("forward: decay dropped from S'", "Sp[a * V + c] = e * S[a * V + c];", "Sp[a * V + c] = S[a * V + c];"),
    ("forward: sign of the delta correction", "u[c] -= Sp[a * V + c] * ka;", "u[c] += Sp[a * V + c] * ka;"),
    ("forward: beta dropped from the write", "double bk = bt * kt[a];", "double bk = kt[a];"),
    ("forward: scale dropped from o", "for (int c = 0; c < V; ++c) ot[c] *= J->scale;", "(void)0;"),
    # backward
    ("backward: scale dropped from dq", "dqt[a] += J->scale * acc;", "dqt[a] += acc;"),
    ("backward: output term dropped from dS", "dS[a * V + c] += sq * dot[c];", "(void)sq;"),
    ("backward: q instead of k in du", "du[c] += dS[a * V + c] * kt[a];", "du[c] += dS[a * V + c] * qt[a];"),
    ("backward: beta dropped from du", "for (int c = 0; c < V; ++c) du[c] *= bt;", "(void)0;"),
    ("backward: sign of S' du in dk", "dkt[a] += bt * dSu[a] - acc;", "dkt[a] += bt * dSu[a] + acc;"),
    ("backward: q instead of k in dbeta", "for (int a = 0; a < K; ++a) db += kt[a] * dSu[a];",
     "for (int a = 0; a < K; ++a) db += qt[a] * dSu[a];"),
    ("backward: sign of k du^T in dS'", "dS[a * V + c] -= kt[a] * du[c];", "dS[a * V + c] += kt[a] * du[c];"),
    ("backward: S_{t-1} instead of S' in dg", "acc += dS[a * V + c] * Sp[a * V + c];",
     "acc += dS[a * V + c] * Sold[a * V + c];"),
    ("backward: decay dropped from dS", "for (int c = 0; c < V; ++c) dS[a * V + c] *= e;", "(void)e;"),
]


def _build(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-D_GNU_SOURCE", "-o", str(so), str(src),
                           "-lm", "-lpthread"])
    lib = ctypes.CDLL(str(so))
    P = ctypes.c_void_p
    lib.kda_oracle_run.restype = ctypes.c_int
    lib.kda_oracle_run.argtypes = [ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_double] + [P] * 18 + [ctypes.c_int]
    lib.kda_oracle_num_chunks.restype = ctypes.c_int64
    lib.kda_oracle_num_chunks.argtypes = [P, ctypes.c_int, ctypes.c_int]
    return lib


@pytest.fixture(scope="module")
def reference():
    # two key heads of two value heads each (a wrong head map shows), h0 and dht present
    inp = kda_inputs.small(seed=5, B=1, T=24, H=2, HV=4, K=4, V=3, dtype="f32")
    x = _f64_inputs(inp)
    assert x["h0"] is not None and x["dht"] is not None
    return x, _torch_literal(x, 2)


def _worst_error(lib, monkeypatch, x, ref):
    monkeypatch.setattr(oracle, "_lib", lib)
    r = oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], x["do"], x["dht"], x["cu"],
                   chunk=8)
    return max(np.linalg.norm(r[key] - val) / max(np.linalg.norm(val), 1e-300) for key, val in ref.items())


def test_unmodified_source_meets_the_pin(tmp_path, monkeypatch, reference):
    x, ref = reference
    with open(SRC) as f:
        text = f.read()
    assert _worst_error(_build(tmp_path, "control", text), monkeypatch, x, ref) < 1e-12


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, monkeypatch, reference, name, old, new):
    x, ref = reference
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, name
    err = _worst_error(_build(tmp_path, "mutant", text.replace(old, new)), monkeypatch, x, ref)
    assert err > 1e-6, (name, err)


CHUNKED_SRC = os.path.join(os.path.dirname(oracle.__file__), "chunked.py")

CHUNKED_MUTANTS = [
    ("beta of the column in Akk", "Akk = bc[:, None] * M", "Akk = bc[None, :] * M"),
    ("Aqk mask drops the diagonal", 'Aqk = scale * np.einsum("rd,jd,rjd->rj", qc, kc, D) * _tri(c, False)',
     'Aqk = scale * np.einsum("rd,jd,rjd->rj", qc, kc, D) * _tri(c, True)'),
    ("K^ decay reversed", "Kh = kc * np.exp(GamC[None, :] - Gam)", "Kh = kc * np.exp(Gam - GamC[None, :])"),
    ("Aqk not transposed in d_delta", "d_delta = Aqk.T @ dO + Kh @ dS_out", "d_delta = Aqk @ dO + Kh @ dS_out"),
    ("triangle backward not transposed", "dAkk = -(INV.T @ dINV @ INV.T) * _tri(c, True)",
     "dAkk = -(INV @ dINV @ INV) * _tri(c, True)"),
    ("Akk term dropped from dbeta", "dbeta += np.sum(dAkk * M, axis=1)", "pass"),
    ("sign of the K^ term in dGamma", "dGam -= dKh * Kh", "dGam += dKh * Kh"),
    ("Gamma_C terms dropped", "dGam[-1] += dGamC", "pass"),
]


def _load_chunked(tmp_path, name, text):
    path = tmp_path / f"{name}.py"
    path.write_text(text.replace("from . import _f64", "from oracle import _f64"))
    spec = importlib.util.spec_from_file_location(f"chunked_{name}", str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="module")
def recurrence():
    inp = kda_inputs.small(seed=6, B=1, T=0, H=1, HV=2, K=8, V=8, dtype="f32", seq_lens=[19, 40])
    return inp, oracle.run_inputs(inp, chunk=16, chunk_states=True)


def _chunked_error(mod, inp, ref):
    b = mod.run_chunked(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, inp.h0, inp.do, inp.dht, inp.cu_seqlens,
                        chunk=16)
    keys = ["o", "ht", "s_in", "ds_out", "dq", "dk", "dv", "dg", "dbeta", "dh0"]
    return max(np.abs(b[k] - ref[k]).max() / max(np.abs(ref[k]).max(), 1e-300) for k in keys)


def test_unmodified_chunked_form_meets_the_pin(tmp_path, recurrence):
    inp, ref = recurrence
    with open(CHUNKED_SRC) as f:
        text = f.read()
    assert _chunked_error(_load_chunked(tmp_path, "control", text), inp, ref) < 1e-12


@pytest.mark.parametrize("name,old,new", CHUNKED_MUTANTS, ids=[m[0] for m in CHUNKED_MUTANTS])
def test_planted_mistake_in_chunked_form_is_caught(tmp_path, recurrence, name, old, new):
    inp, ref = recurrence
    with open(CHUNKED_SRC) as f:
        text = f.read()
    assert text.count(old) == 1, name
    err = _chunked_error(_load_chunked(tmp_path, "mutant", text.replace(old, new)), inp, ref)
    assert err > 1e-6, (name, err)
