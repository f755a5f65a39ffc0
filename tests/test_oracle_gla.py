"""Pins of the oracle's gated (per-key decay) form, against things other than
the oracle itself.

Reading (the ejkernel `recurrent` gate g, GLA-style, with the keys' shape):
token t decays row a of the state by exp(g_gamma[h] + g_t[a]) before adding
k_t v_t^T.  Pins:
  * a brute-force quadratic form written from that definition (products of
    decays between every pair of tokens), forward and final state;
  * finite differences of sum(o*do) + sum(final*dfinal) for every gradient,
    dg included;
  * a gate constant per head reduces to the ungated recurrence with g_gamma
    shifted by that constant;
  * the identity the GPU path uses for dg (log-decay cumulative sums G_t):
    dG_t = q_t*dq_t - k_t*dk_t (+ sum_b F*dF at the last token),
    dg = reverse cumulative sum of dG over the processing order.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def _problem(B=2, T=7, H=2, d=3, e=2, seed=0, strong=False):
    r = np.random.default_rng(seed)
    q, k, v, do = (r.standard_normal((B, T, H, x)) for x in (d, d, e, e))
    g = -(r.random((B, T, H, d)) * (2.0 if strong else 0.5))
    gg = -r.random(H) * 0.3
    s0 = r.standard_normal((B, H, d, e)) * 0.5
    dfin = r.standard_normal((B, H, d, e)) * 0.5
    return q, k, v, do, g, gg, s0, dfin


def _brute(q, k, v, g, gg, scale, s0, reverse):
    """o and final state from the definition: pairwise decay products."""
    B, T, H, d = q.shape
    e = v.shape[3]
    o = np.zeros((B, T, H, e))
    fin = np.zeros((B, H, d, e))
    order = list(range(T))[::-1] if reverse else list(range(T))
    for b in range(B):
        for h in range(H):
            dec = np.exp(gg[h] + g[b, :, h, :])          # [T, d]
            for pi, t in enumerate(order):
                acc = np.zeros(e)
                for pj in range(pi + 1):
                    u = order[pj]
                    w = np.prod(dec[[order[x] for x in range(pj + 1, pi + 1)]], axis=0) \
                        if pj < pi else np.ones(d)
                    acc += (q[b, t, h] * k[b, u, h] * w).sum() * v[b, u, h]
                wall = np.prod(dec[[order[x] for x in range(pi + 1)]], axis=0)
                acc += (q[b, t, h] * wall) @ s0[b, h]
                o[b, t, h] = scale * acc
            wall = np.prod(dec, axis=0)
            f = wall[:, None] * s0[b, h]
            for pj, u in enumerate(order):
                w = np.prod(dec[[order[x] for x in range(pj + 1, T)]], axis=0) \
                    if pj < T - 1 else np.ones(d)
                f += np.outer(w * k[b, u, h], v[b, u, h])
            fin[b, h] = f
    return o, fin


@pytest.mark.parametrize("reverse", [False, True])
def test_gated_forward_matches_brute_force(reverse):
    q, k, v, do, g, gg, s0, dfin = _problem(seed=1)
    o, fin = oracle.gla_forward(q, k, v, g, gg, 0.7, s0, reverse)
    ob, fb = _brute(q, k, v, g, gg, 0.7, s0, reverse)
    np.testing.assert_allclose(o, ob, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(fin, fb, rtol=1e-10, atol=1e-12)


def test_constant_gate_is_a_shifted_g_gamma():
    q, k, v, do, g, gg, s0, dfin = _problem(seed=2)
    c = np.array([-0.25, -0.6])
    gate = np.broadcast_to(c[None, None, :, None], g.shape).copy()
    o1, f1 = oracle.gla_forward(q, k, v, gate, gg, 0.5, s0)
    o2, f2 = oracle.forward(q, k, v, gg + c, 0.5, s0)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(f1, f2, rtol=1e-12, atol=1e-13)
    g1 = oracle.gla_backward(q, k, v, gate, gg, 0.5, do, s0, dfin)
    g2 = oracle.backward(q, k, v, gg + c, 0.5, do, s0, dfin)
    for a, b in zip((g1[0], g1[1], g1[2], g1[4]), g2):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def _loss(q, k, v, g, gg, scale, s0, do, dfin, reverse, cu=None):
    o, fin = oracle.gla_forward(q, k, v, g, gg, scale, s0, reverse, cu)
    return float((o * do).sum() + (fin * dfin).sum())


@pytest.mark.parametrize("reverse", [False, True])
def test_gated_gradients_match_finite_differences(reverse):
    q, k, v, do, g, gg, s0, dfin = _problem(B=1, T=6, H=1, d=3, e=2, seed=3, strong=True)
    dq, dk, dv, dg, ds0 = oracle.gla_backward(q, k, v, g, gg, 0.8, do, s0, dfin, reverse)
    args = dict(q=q, k=k, v=v, g=g, s0=s0)
    grads = dict(q=dq, k=dk, v=dv, g=dg, s0=ds0)
    eps = 1e-6
    for name, x in args.items():
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            a1 = dict(args, **{name: xp})
            a2 = dict(args, **{name: xm})
            num[idx] = (_loss(a1["q"], a1["k"], a1["v"], a1["g"], gg, 0.8, a1["s0"], do, dfin,
                              reverse)
                        - _loss(a2["q"], a2["k"], a2["v"], a2["g"], gg, 0.8, a2["s0"], do, dfin,
                                reverse)) / (2 * eps)
        np.testing.assert_allclose(grads[name], num, rtol=1e-6, atol=1e-7, err_msg=name)


@pytest.mark.parametrize("reverse", [False, True])
def test_dg_identity_from_dq_dk(reverse):
    B, T, H, d, e = 2, 9, 2, 4, 3
    q, k, v, do, g, gg, s0, dfin = _problem(B, T, H, d, e, seed=4)
    dq, dk, dv, dg, ds0 = oracle.gla_backward(q, k, v, g, gg, 0.6, do, s0, dfin, reverse)
    _, fin = oracle.gla_forward(q, k, v, g, gg, 0.6, s0, reverse)
    dG = q * dq - k * dk                                  # [B, T, H, d]
    order = np.arange(T)[::-1] if reverse else np.arange(T)
    last = order[-1]
    dG[:, last] += np.einsum("bhde,bhde->bhd", fin, dfin)
    ident = np.zeros_like(dG)
    run = np.zeros((B, H, d))
    for t in order[::-1]:                                 # reverse of processing order
        run = run + dG[:, t]
        ident[:, t] = run
    np.testing.assert_allclose(dg, ident, rtol=1e-9, atol=1e-11)


def test_gated_packed_sequences_are_independent():
    q, k, v, do, g, gg, s0, dfin = _problem(B=1, T=9, H=2, d=3, e=2, seed=5)
    cu = np.array([0, 4, 4, 9], dtype=np.int32)
    s0p = np.concatenate([s0, -s0, 0.5 * s0], 0)
    o, fin = oracle.gla_forward(q, k, v, g, gg, 0.5, s0p, False, cu)
    for n, (a, b) in enumerate(((0, 4), (4, 4), (4, 9))):
        oa, fa = oracle.gla_forward(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], gg, 0.5,
                                    s0p[n:n + 1])
        np.testing.assert_allclose(o[:, a:b], oa, rtol=1e-12)
        np.testing.assert_allclose(fin[n:n + 1], fa, rtol=1e-12)
