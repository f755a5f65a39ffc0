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
    ("wrong_decay_sign", "exp(J->g_gamma[h])", "exp(-J->g_gamma[h])", 0),
    ("dropped_initial_state", "memcpy(S, J->init + sidx, sizeof(double) * d * e);",
     "memset(S, 0, sizeof(double) * d * e);", 0),
    ("ignored_reverse_fwd", "J->reverse ? len - 1 - step : step", "step", 0),
    ("read_before_update", "S[a * e + b] = gamma * S[a * e + b] + kt[a] * vt[b];",
     "S[a * e + b] = S[a * e + b] + kt[a] * vt[b] * gamma;", 0),
    ("dq_missing_scale", "dqt[a] = J->scale * acc;", "dqt[a] = acc;", 0),
    ("dropped_bwd_decay", "G[a] *= gamma;", "G[a] *= 1.0;", 0),
    ("dv_wrong_operand", "acc += G[a * e + b] * kt[a];", "acc += G[a * e + b] * qt[a];", 0),
    ("dk_transposed_state", "acc += G[a * e + b] * vt[b];", "acc += G[b * e + a % e] * vt[b];", 0),
    ("dropped_dfinal", "memcpy(G, J->dfinal + sidx, sizeof(double) * d * e);",
     "memset(G, 0, sizeof(double) * d * e);", 0),
    ("ignored_reverse_bwd", "J->reverse ? len - 1 - step : step", "step", 2),
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
    for fn in ("la_oracle_fwd", "la_oracle_bwd"):
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
