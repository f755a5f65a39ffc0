"""Pins for the fp64 CPU oracle (oracle/): nothing here runs on a GPU.

Each test checks the oracle against something other than itself:
  * the brute-force quadratic form (tests/brute_force.py), a different
    formulation of the same recurrence (d != e so a transposed operand fails);
  * closed forms: all-ones inputs (the docstring examples of the ejkernel
    lightning_attn and recurrent pages), gamma = 0, T = 1, g = 0 as a cumsum;
  * d = e = 1, where the recurrence is a first-order IIR filter, against
    scipy.signal.lfilter;
  * invariants: split run with state hand-off, reverse = flip-run-flip,
    packed varlen = per-sequence runs;
  * central finite differences of sum(o*do) + sum(final*dF) for every gradient.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from brute_force import brute
from workloads import random_small, lightning_g_gamma

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def _problem(seed, B=2, T=13, H=3, d=5, e=4, with_init=True, with_dF=True):
    p = random_small(seed, B, T, H, d, e)
    rng = np.random.default_rng(seed + 1000)
    init = rng.standard_normal((B, H, d, e)) if with_init else None
    dF = rng.standard_normal((B, H, d, e)) if with_dF else None
    return (p["q"].numpy(), p["k"].numpy(), p["v"].numpy(), p["do"].numpy(),
            p["g_gamma"].numpy(), init, dF)


@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_forward_matches_brute_force(seed, reverse):
    q, k, v, do, g, init, dF = _problem(seed)
    o, fin = oracle.forward(q, k, v, g, 0.7, init, reverse)
    ob, finb = brute(q, k, v, g, 0.7, init, reverse)
    assert _rel(o, ob) < 1e-12
    assert _rel(fin, finb) < 1e-12


@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("seed", [3, 4])
def test_backward_matches_brute_force(seed, reverse):
    q, k, v, do, g, init, dF = _problem(seed)
    got = oracle.backward(q, k, v, g, 1.3, do, init, dF, reverse)
    ref = brute(q, k, v, g, 1.3, init, reverse, do=do, d_final_state=dF)[2:]
    for a, b in zip(got, ref):
        assert _rel(a, b) < 1e-12


def test_backward_without_optional_state_matches_brute_force():
    q, k, v, do, g, _, _ = _problem(5, with_init=False, with_dF=False)
    got = oracle.backward(q, k, v, g, 0.5, do)
    ref = brute(q, k, v, g, 0.5, do=do)[2:]
    for a, b in zip(got, ref):
        assert _rel(a, b) < 1e-12


def _loss(q, k, v, g, s, init, reverse, do, dF, cu=None):
    o, fin = oracle.forward(q, k, v, g, s, init, reverse, cu)
    return float(np.sum(o * do) + np.sum(fin * dF))


@pytest.mark.parametrize("reverse", [False, True])
def test_gradients_match_finite_differences(reverse):
    q, k, v, do, g, init, dF = _problem(7, B=1, T=6, H=2, d=3, e=2)
    s = 0.9
    dq, dk, dv, dinit = oracle.backward(q, k, v, g, s, do, init, dF, reverse)
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv), ("init", init, dinit)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args = dict(q=q, k=k, v=v, init=init)
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], g, s, args["init"], reverse, do, dF)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], g, s, args["init"], reverse, do, dF)
            fd[idx] = (lp - lm) / (2 * eps)
        assert _rel(grad, fd) < 1e-7, name


def test_varlen_gradients_match_finite_differences():
    q, k, v, do, g, _, _ = _problem(8, B=1, T=9, H=2, d=3, e=2, with_init=False, with_dF=False)
    cu = np.array([0, 4, 4, 9], dtype=np.int32)
    rng = np.random.default_rng(8)
    init = rng.standard_normal((3, 2, 3, 2))
    dF = rng.standard_normal((3, 2, 3, 2))
    s = 1.1
    dq, dk, dv, dinit = oracle.backward(q, k, v, g, s, do, init, dF, True, cu)
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv), ("init", init, dinit)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            vals = []
            for sgn in (1, -1):
                xx = x.copy(); xx[idx] += sgn * eps
                args = dict(q=q, k=k, v=v, init=init)
                args[name] = xx
                vals.append(_loss(args["q"], args["k"], args["v"], g, s, args["init"], True,
                                  do, dF, cu))
            fd[idx] = (vals[0] - vals[1]) / (2 * eps)
        assert _rel(grad, fd) < 1e-7, name


def _all_ones_closed_form(T, d, g, s):
    """All-ones q,k,v, zero state: o_t[:] = s*d*sum_{u<=t} gamma^(t-u), final[:,:] =
    sum_u gamma^(T-1-u) -- geometric sums."""
    gam = math.exp(g)
    t = np.arange(T, dtype=np.float64)
    if gam == 1.0:
        return s * d * (t + 1), float(T)
    return s * d * (1 - gam ** (t + 1)) / (1 - gam), (1 - gam ** T) / (1 - gam)


def test_all_ones_lightning_example_closed_form():
    # ejkernel lightning_attn module docstring, Example: (2, 2048, 8, 64) ones,
    # layer_idx=5, num_layers=12, default scale 1/sqrt(head_dim).
    B, T, H, d = 2, 2048, 8, 64
    ones = np.ones((B, T, H, d))
    g = lightning_g_gamma(H, 5, 12).numpy().astype(np.float64)
    s = d ** -0.5
    o, fin = oracle.forward(ones, ones, ones, g, s)
    assert o.shape == (B, T, H, d) and fin.shape == (B, H, d, d)
    for h in range(H):
        o_ref, f_ref = _all_ones_closed_form(T, d, g[h], s)
        assert _rel(o[:, :, h, :], np.broadcast_to(o_ref[None, :, None], (B, T, d))) < 1e-12
        assert np.allclose(fin[:, h], f_ref, rtol=1e-12, atol=0)


def test_all_ones_recurrent_example_closed_form():
    # ejkernel recurrent docstring, Examples: (2, 100, 8, 64) ones with
    # g_gamma = -arange(8) * 0.1.
    B, T, H, d = 2, 100, 8, 64
    ones = np.ones((B, T, H, d))
    g = -np.arange(8, dtype=np.float32).astype(np.float64) * 0.1
    s = 1.0 / math.sqrt(d)
    o, fin = oracle.forward(ones, ones, ones, g, s)
    for h in range(H):
        o_ref, f_ref = _all_ones_closed_form(T, d, g[h], s)
        assert _rel(o[0, :, h, 0], o_ref) < 1e-12
        assert np.allclose(fin[:, h], f_ref, rtol=1e-12, atol=0)


def test_page_shape_examples():
    """Shapes printed on the pages (tests/golden/page_examples.json)."""
    with open(os.path.join(GOLDEN, "page_examples.json")) as f:
        ex = json.load(f)
    r = ex["recurrent_varlen"]
    T, H, d = r["q_shape"]
    ones = np.ones((1, T, H, d))
    cu = np.array(r["cu_seqlens"], dtype=np.int32)
    o, fin = oracle.forward(ones, ones, ones, np.zeros(H), d ** -0.5, cu_seqlens=cu)
    assert list(o.shape[1:]) == r["o_shape"]
    assert list(fin.shape) == r["final_state_shape"]
    r = ex["recurrent_dense"]
    B, T, H, d = r["q_shape"]
    ones = np.ones((B, T, H, d))
    o, fin = oracle.forward(ones, ones, ones, np.zeros(H), d ** -0.5)
    assert list(o.shape) == r["o_shape"]
    # each packed sequence restarts from zero: with g = 0 and all ones the output
    # of the first token of every sequence is s*d.
    o, _ = oracle.forward(np.ones((1, 150, 2, 4)), np.ones((1, 150, 2, 4)),
                          np.ones((1, 150, 2, 4)), np.zeros(2), 0.5, cu_seqlens=cu)
    for start in r_varlen_starts(ex):
        assert np.allclose(o[0, start], 0.5 * 4)


def r_varlen_starts(ex):
    return ex["recurrent_varlen"]["cu_seqlens"][:-1]


def test_gamma_zero_is_diagonal_only():
    q, k, v, do, g, init, dF = _problem(11)
    g = np.full_like(g, -1e4)          # exp(-1e4) == 0 in float64
    o, fin = oracle.forward(q, k, v, g, 0.8, init)
    ref = 0.8 * np.einsum("bthd,bthd->bth", q, k)[..., None] * v
    assert _rel(o, ref) < 1e-13
    ref_fin = np.einsum("bhd,bhe->bhde", k[:, -1], v[:, -1])
    assert _rel(fin, ref_fin) < 1e-13


def test_single_token_closed_form():
    q, k, v, do, g, init, dF = _problem(12, T=1)
    o, fin = oracle.forward(q, k, v, g, 1.7, init)
    gam = np.exp(g)[None, :, None, None]
    S = gam * init + np.einsum("bhd,bhe->bhde", k[:, 0], v[:, 0])
    assert _rel(fin, S) < 1e-13
    assert _rel(o[:, 0], 1.7 * np.einsum("bhd,bhde->bhe", q[:, 0], S)) < 1e-13


def test_no_decay_is_cumulative_sum():
    q, k, v, do, g, init, dF = _problem(13, with_init=False)
    g = np.zeros_like(g)
    o, fin = oracle.forward(q, k, v, g, 0.6)
    kv = np.cumsum(np.einsum("bthd,bthe->bthde", k, v), axis=1)
    ref = 0.6 * np.einsum("bthd,bthde->bthe", q, kv)
    assert _rel(o, ref) < 1e-12
    assert _rel(fin, kv[:, -1]) < 1e-12


@pytest.mark.parametrize("reverse", [False, True])
def test_scalar_state_is_first_order_iir_filter(reverse):
    scipy_signal = pytest.importorskip("scipy.signal")
    q, k, v, do, g, init, dF = _problem(14, B=1, T=40, H=2, d=1, e=1)
    o, fin = oracle.forward(q, k, v, g, 1.0, init, reverse)
    for h in range(2):
        x = (k[0, :, h, 0] * v[0, :, h, 0])
        gam = math.exp(g[h])
        if reverse:
            x = x[::-1]
        zi = np.array([gam * init[0, h, 0, 0]])
        y, _ = scipy_signal.lfilter([1.0], [1.0, -gam], x, zi=zi)
        if reverse:
            y = y[::-1]
        assert _rel(o[0, :, h, 0], q[0, :, h, 0] * y) < 1e-12
        assert abs(fin[0, h, 0, 0] - (y[-1] if not reverse else y[0])) < 1e-12 * max(1, abs(y).max())


def test_split_run_hands_off_state():
    q, k, v, do, g, init, dF = _problem(15, T=20)
    o, fin = oracle.forward(q, k, v, g, 1.0, init)
    o1, f1 = oracle.forward(q[:, :7], k[:, :7], v[:, :7], g, 1.0, init)
    o2, f2 = oracle.forward(q[:, 7:], k[:, 7:], v[:, 7:], g, 1.0, f1)
    assert _rel(np.concatenate([o1, o2], axis=1), o) < 1e-13
    assert _rel(f2, fin) < 1e-13
    # gradients chain the same way: d_initial_state of the tail is d_final of the head
    g_full = oracle.backward(q, k, v, g, 1.0, do, init, dF)
    t2 = oracle.backward(q[:, 7:], k[:, 7:], v[:, 7:], g, 1.0, do[:, 7:], f1, dF)
    t1 = oracle.backward(q[:, :7], k[:, :7], v[:, :7], g, 1.0, do[:, :7], init, t2[3])
    for i in range(3):
        assert _rel(np.concatenate([t1[i], t2[i]], axis=1), g_full[i]) < 1e-12
    assert _rel(t1[3], g_full[3]) < 1e-12


def test_reverse_is_flip_run_flip():
    q, k, v, do, g, init, dF = _problem(16)
    o, fin = oracle.forward(q, k, v, g, 0.9, init, reverse=True)
    fl = lambda x: x[:, ::-1].copy()
    of, finf = oracle.forward(fl(q), fl(k), fl(v), g, 0.9, init)
    assert _rel(o, fl(of)) < 1e-13
    assert _rel(fin, finf) < 1e-13
    gr = oracle.backward(q, k, v, g, 0.9, do, init, dF, reverse=True)
    gf = oracle.backward(fl(q), fl(k), fl(v), g, 0.9, fl(do), init, dF)
    for i in range(3):
        assert _rel(gr[i], fl(gf[i])) < 1e-13
    assert _rel(gr[3], gf[3]) < 1e-13


@pytest.mark.parametrize("reverse", [False, True])
def test_varlen_equals_per_sequence_runs(reverse):
    lens = [5, 0, 11, 1, 7]
    cu = np.cumsum([0] + lens).astype(np.int32)
    T = int(cu[-1])
    q, k, v, do, g, _, _ = _problem(17, B=1, T=T, H=2, d=4, e=3, with_init=False,
                                    with_dF=False)
    rng = np.random.default_rng(17)
    init = rng.standard_normal((len(lens), 2, 4, 3))
    dF = rng.standard_normal((len(lens), 2, 4, 3))
    o, fin = oracle.forward(q, k, v, g, 1.2, init, reverse, cu)
    grads = oracle.backward(q, k, v, g, 1.2, do, init, dF, reverse, cu)
    for n, L in enumerate(lens):
        a, b = cu[n], cu[n + 1]
        sl = lambda x: x[:, a:b]
        if L == 0:
            assert np.array_equal(fin[n], init[n])
            assert np.array_equal(grads[3][n], dF[n])
            continue
        o1, f1 = oracle.forward(sl(q), sl(k), sl(v), g, 1.2, init[n:n + 1], reverse)
        g1 = oracle.backward(sl(q), sl(k), sl(v), g, 1.2, sl(do), init[n:n + 1],
                             dF[n:n + 1], reverse)
        assert _rel(o[:, a:b], o1) < 1e-13
        assert _rel(fin[n:n + 1], f1) < 1e-13
        for i in range(3):
            assert _rel(grads[i][:, a:b], g1[i]) < 1e-13
        assert _rel(grads[3][n:n + 1], g1[3]) < 1e-13


def test_thread_count_does_not_change_result():
    q, k, v, do, g, init, dF = _problem(18, B=3, T=30, H=4)
    a = oracle.backward(q, k, v, g, 1.0, do, init, dF, threads=1)
    b = oracle.backward(q, k, v, g, 1.0, do, init, dF, threads=5)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_rejects_bad_arguments():
    q = np.zeros((2, 4, 1, 2))
    with pytest.raises(ValueError):
        oracle.forward(q, q, q, [0.0], 1.0, cu_seqlens=[0, 4])        # batch != 1
    with pytest.raises(ValueError):
        oracle.forward(q[:1], q[:1], q[:1], [0.0], 1.0, cu_seqlens=[0, 3])  # last != T
    with pytest.raises(ValueError):
        oracle.forward(q, q, q, [0.0], 1.0, initial_state=np.zeros((3, 1, 2, 2)))
