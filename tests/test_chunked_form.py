"""The chunked form the CUDA sweeps evaluate, restated in numpy from its
derivation (a chunk's decay-masked scores, the inter-chunk term read from the
entry state, the state carried with gamma^Lc, and the backward's G = dL/dS
carried against processing order), checked against the fp64 oracle's
token-by-token recurrence for several chunk sizes, both directions, packed
sequences and strong decay.  This pins the algebra the kernels are built on;
it shares nothing with them."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _decay_mask(gamma, Lc):
    p = np.arange(Lc)
    m = p[:, None] - p[None, :]
    return np.where(m >= 0, gamma ** np.maximum(m, 0), 0.0), p


def chunked_forward(q, k, v, gamma, s, S0, C, reverse):
    """One (sequence, head): q, k [L, d], v [L, e], S0 [d, e]."""
    L = q.shape[0]
    order = np.arange(L)[::-1] if reverse else np.arange(L)
    o = np.zeros((L, v.shape[1]))
    S = S0.copy()
    for c0 in range(0, L, C):
        idx = order[c0:c0 + C]
        Lc = len(idx)
        Q, K, V = q[idx], k[idx], v[idx]
        D, p = _decay_mask(gamma, Lc)
        P = s * (Q @ K.T) * D
        o[idx] = P @ V + s * (gamma ** (p + 1))[:, None] * (Q @ S)
        S = gamma ** Lc * S + (K * (gamma ** (Lc - 1 - p))[:, None]).T @ V
    return o, S


def chunked_backward(q, k, v, do, gamma, s, S0, dF, C, reverse):
    L = q.shape[0]
    order = np.arange(L)[::-1] if reverse else np.arange(L)
    dq, _ = chunked_forward(do, v, k, gamma, s, S0.T, C, reverse)
    dk, dv = np.zeros_like(k), np.zeros_like(v)
    G = dF.copy()
    starts = list(range(0, L, C))
    for c0 in reversed(starts):
        idx = order[c0:c0 + C]
        Lc = len(idx)
        Q, K, V, DO = q[idx], k[idx], v[idx], do[idx]
        D, p = _decay_mask(gamma, Lc)
        tail = (gamma ** (Lc - 1 - p))[:, None]
        A = s * (Q @ K.T) * D             # A_ij: query i (later), key j
        Bm = s * (DO @ V.T) * D
        dv[idx] = A.T @ DO + tail * (K @ G)
        dk[idx] = Bm.T @ Q + tail * (V @ G.T)
        G = gamma ** Lc * G + s * (Q * (gamma ** (p + 1))[:, None]).T @ DO
    return dq, dk, dv, G


def _run_all(x, C, reverse):
    q, k, v, do = (x[n].numpy() for n in ("q", "k", "v", "do"))
    g = x["g_gamma"].numpy().astype(np.float64)
    init, dfin = x["initial_state"].numpy(), x["d_final_state"].numpy()
    cu = x["cu_seqlens"]
    spans = ([(b, 0, q.shape[1], b) for b in range(q.shape[0])] if cu is None else
             [(0, int(cu[n]), int(cu[n + 1]), n) for n in range(len(cu) - 1)])
    out = {n: np.zeros_like(t) for n, t in (("o", v), ("dq", q), ("dk", k), ("dv", v))}
    fin, dinit = np.zeros_like(init), np.zeros_like(init)
    for row, a, b, n in spans:
        for h in range(q.shape[2]):
            sl = (row, slice(a, b), h)
            gamma = np.exp(g[h])
            o, S = chunked_forward(q[sl], k[sl], v[sl], gamma, x["scale"], init[n, h], C, reverse)
            dq, dk, dv, G = chunked_backward(q[sl], k[sl], v[sl], do[sl], gamma, x["scale"],
                                             init[n, h], dfin[n, h], C, reverse)
            out["o"][sl], out["dq"][sl], out["dk"][sl], out["dv"][sl] = o, dq, dk, dv
            fin[n, h], dinit[n, h] = S, G
    out.update(final_state=fin, d_initial_state=dinit)
    return out


def _oracle_all(x, reverse):
    o, fin = oracle.forward(x["q"], x["k"], x["v"], x["g_gamma"], x["scale"],
                            x["initial_state"], reverse, x["cu_seqlens"])
    dq, dk, dv, dinit = oracle.backward(x["q"], x["k"], x["v"], x["g_gamma"], x["scale"],
                                        x["do"], x["initial_state"], x["d_final_state"],
                                        reverse, x["cu_seqlens"])
    return dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, d_initial_state=dinit)


def _assert_close(got, ref, tol=1e-10):
    for name, r in ref.items():
        r = np.asarray(r, dtype=np.float64)
        err = np.max(np.abs(got[name] - r)) / max(np.max(np.abs(r)), 1e-300)
        assert err <= tol, (name, err)


@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("reverse", [False, True])
def test_chunked_form_equals_the_recurrence(C, reverse):
    x = W.random_small(5, 2, 37, 3, 5, 4, g_lo=-1.5, g_hi=0.0)
    x["g_gamma"][0] = 0.0                                   # a head without decay
    gen = np.random.default_rng(1)
    x["initial_state"] = torch.as_tensor(gen.standard_normal((2, 3, 5, 4)))
    x["d_final_state"] = torch.as_tensor(gen.standard_normal((2, 3, 5, 4)))
    x["scale"], x["cu_seqlens"] = 0.7, None
    _assert_close(_run_all(x, C, reverse), _oracle_all(x, reverse))


@pytest.mark.parametrize("reverse", [False, True])
def test_chunked_form_packed_and_strong_decay(reverse):
    # packed sequences (one empty), a chunk size that leaves ragged chunks, and a
    # decay of exp(-40) per token: every factor stays a non-negative power of gamma
    x = W.random_small(9, 1, 41, 2, 4, 6, g_lo=-40.0, g_hi=-0.01)
    gen = np.random.default_rng(2)
    x["initial_state"] = torch.as_tensor(gen.standard_normal((4, 2, 4, 6)))
    x["d_final_state"] = torch.as_tensor(gen.standard_normal((4, 2, 4, 6)))
    x["scale"], x["cu_seqlens"] = 0.5, [0, 9, 9, 30, 41]
    _assert_close(_run_all(x, 8, reverse), _oracle_all(x, reverse))
