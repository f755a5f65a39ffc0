"""Planted mistakes: each mutant is a copy of oracle/la_oracle.c with one
plausible error (a transposed operand, a dropped term, a wrong sign, an
ignored flag), compiled on the CPU into a temporary library.  The test checks
that the oracle's pins (brute-force quadratic form, forward and backward, both
directions, with initial and final states) reject every mutant, and accept the
unmodified source compiled the same way.  The oracle source is never changed.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from brute_force import brute
from workloads import random_small

SRC = os.path.join(os.path.dirname(oracle.__file__), "la_oracle.c")

# (name, exact text in la_oracle.c, replacement, occurrence to replace (0-based))
MUTANTS = [
    ("transposed_kv_outer", "kt[a] * vt[b];", "kt[b % d] * vt[a % e];", 0),
    ("dropped_scale", "ot[b] = J->scale * acc;", "ot[b] = acc;", 0),
    ("wrong_decay_sign", ": exp(gh);", ": exp(-gh);", 0),
    ("dropped_initial_state", "memcpy(S, J->init + sidx, sizeof(double) * d * e);",
     "memset(S, 0, sizeof(double) * d * e);", 0),
    ("ignored_reverse_fwd", "J->reverse ? len - 1 - step : step", "step", 0),
    ("read_before_update", "S[a * e + b] = da * S[a * e + b] + kt[a] * vt[b];",
     "S[a * e + b] = S[a * e + b] + kt[a] * vt[b] * da;", 0),
    ("dq_missing_scale", "dqt[a] = J->scale * acc;", "dqt[a] = acc;", 0),
    ("dropped_bwd_decay", "G[a * e + b] *= da;", "G[a * e + b] *= 1.0;", 0),
    ("dv_wrong_operand", "acc += G[a * e + b] * kt[a];", "acc += G[a * e + b] * qt[a];", 0),
    ("dk_transposed_state", "acc += G[a * e + b] * vt[b];", "acc += G[b * e + a % e] * vt[b];", 0),
    ("dropped_dfinal", "memcpy(G, J->dfinal + sidx, sizeof(double) * de);",
     "memset(G, 0, sizeof(double) * de);", 0),
    ("ignored_reverse_bwd", "J->reverse ? len - 1 - step : step", "step", 2),
]

# Mutants of the gated (per-key decay) form, checked by the gated pins.
GATED_MUTANTS = [
    ("dg_missing_decay", "dgt[a] = decay(J, row, t, h, a, gh) * acc;", "dgt[a] = acc;", 0),
    ("gate_of_first_channel", "const double da = decay(J, row, t, h, a, gh);",
     "const double da = decay(J, row, t, h, 0, gh);", 0),
    ("dg_uses_next_state", "const double *prev = blk + (step % K) * de;",
     "const double *prev = blk + ((step + 1) % K) * de;", 0),
]


def _compile(tmp_path, name, text):
    src = tmp_path / (name + ".c")
    src.write_text(text)
    lib = tmp_path / ("lib" + name + ".so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-D_POSIX_C_SOURCE=200809L",
                    str(src), "-o", str(lib), "-lm", "-lpthread"], check=True)
    return str(lib)


def _bind(path, monkeypatch):
    real = oracle._load()
    lib = ctypes.CDLL(path)
    for fn in ("la_oracle_fwd", "la_oracle_bwd", "la_oracle_gla_fwd", "la_oracle_gla_bwd"):
        getattr(lib, fn).restype = getattr(real, fn).restype
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
    monkeypatch.setattr(oracle, "_lib", lib)


def _pins_pass():
    """True when the bound library agrees with the brute force on every case."""
    for seed, reverse in ((0, False), (1, True)):
        p = random_small(seed, 2, 9, 2, 4, 3)
        q, k, v, do, g = (p[n].numpy() for n in ("q", "k", "v", "do", "g_gamma"))
        rng = np.random.default_rng(seed)
        init = rng.standard_normal((2, 2, 4, 3))
        dF = rng.standard_normal((2, 2, 4, 3))
        got = oracle.forward(q, k, v, g, 0.7, init, reverse) + \
            oracle.backward(q, k, v, g, 0.7, do, init, dF, reverse)
        ref = brute(q, k, v, g, 0.7, init, reverse, do=do, d_final_state=dF)
        for a, b in zip(got, ref):
            if not np.max(np.abs(a - b)) <= 1e-10 * max(1.0, np.max(np.abs(b))):
                return False
    return True


def test_unmodified_copy_passes(tmp_path, monkeypatch):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    _bind(_compile(tmp_path, "original", open(SRC).read()), monkeypatch)
    assert _pins_pass()


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_rejected(tmp_path, monkeypatch, name, old, new, occ):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    text = open(SRC).read()
    parts = text.split(old)
    assert len(parts) > occ + 1, "mutation site not found: " + old
    mutated = old.join(parts[:occ + 1]) + new + old.join(parts[occ + 1:])
    _bind(_compile(tmp_path, name, mutated), monkeypatch)
    assert not _pins_pass(), name + " slipped through the pins"


def _gated_pins_pass():
    """Gated form: forward against the pairwise-decay brute force of
    test_oracle_gla, and dg against the identity from dq and dk."""
    from test_oracle_gla import _brute, _problem
    for seed, reverse in ((0, False), (1, True)):
        q, k, v, do, g, gg, s0, dfin = _problem(B=2, T=9, H=2, d=4, e=3, seed=seed)
        o, fin = oracle.gla_forward(q, k, v, g, gg, 0.6, s0, reverse)
        ob, fb = _brute(q, k, v, g, gg, 0.6, s0, reverse)
        if not (np.allclose(o, ob, rtol=1e-10, atol=1e-12) and
                np.allclose(fin, fb, rtol=1e-10, atol=1e-12)):
            return False
        dq, dk, dv, dg, ds0 = oracle.gla_backward(q, k, v, g, gg, 0.6, do, s0, dfin, reverse)
        dG = q * dq - k * dk
        order = np.arange(9)[::-1] if reverse else np.arange(9)
        dG[:, order[-1]] += np.einsum("bhde,bhde->bhd", fin, dfin)
        run = np.zeros((2, 2, 4))
        ident = np.zeros_like(dG)
        for t in order[::-1]:
            run = run + dG[:, t]
            ident[:, t] = run
        if not np.allclose(dg, ident, rtol=1e-9, atol=1e-11):
            return False
    return True


def test_unmodified_copy_passes_gated_pins(tmp_path, monkeypatch):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    _bind(_compile(tmp_path, "original_g", open(SRC).read()), monkeypatch)
    assert _gated_pins_pass()


@pytest.mark.parametrize("name,old,new,occ", GATED_MUTANTS, ids=[m[0] for m in GATED_MUTANTS])
def test_gated_mutant_is_rejected(tmp_path, monkeypatch, name, old, new, occ):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    text = open(SRC).read()
    parts = text.split(old)
    assert len(parts) > occ + 1, "mutation site not found: " + old
    mutated = old.join(parts[:occ + 1]) + new + old.join(parts[occ + 1:])
    _bind(_compile(tmp_path, name, mutated), monkeypatch)
    assert not _gated_pins_pass(), name + " slipped through the gated pins"
