"""The gated (per-key gate) chunked form the CUDA path evaluates, restated in
numpy from its derivation and checked against the fp64 oracle's token loop.
Per chunk, in processing order, b holds the running sums of the log-decays
l = g_gamma + g per key channel, B their total, and r = max(midrange(b), -72)
a reference per channel:
  q~ = q e^(b - r), k~ = k e^(r - b);
  o = s [q~ (e^r S) + causal(q~ k~^T) v];  S' = e^(B - r) (e^r S + k~^T v),
the entering state scaled by e^r and the new one by e^(B - r), one after the
other.  Backward: dq~ = dq e^(r - b) from the forward form on (do, v, k~) with
the transposed state; dv from (k~, q~, do) and dk~ = dk e^(b - r) from
(v, do, q~), both carrying H = dL/dS backwards as e^r (s q~^T do + e^(B - r) H);
dg from the identity dL/dG_t = q_t dq_t - k_t dk_t (+ sum_e F dF at the last
token), summed from each token to the end of its sequence.  This pins the
algebra the kernels are built on; it shares nothing with them."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

LIM = 72.0


def _chunks(L, C, reverse):
    order = np.arange(L)[::-1] if reverse else np.arange(L)
    return [order[c0:c0 + C] for c0 in range(0, L, C)]


def _rescale(Q, K, Lg):
    b = np.cumsum(Lg, axis=0)
    r = np.maximum((b.max(0) + b.min(0)) / 2, -LIM)
    return Q * np.exp(b - r), K * np.exp(r - b), b, b[-1], r


def gated_forward(q, k, v, l, s, S0, C, reverse):
    o = np.zeros((q.shape[0], v.shape[1]))
    S = S0.copy()
    for idx in _chunks(q.shape[0], C, reverse):
        Qt, Kt, b, B, r = _rescale(q[idx], k[idx], l[idx])
        mask = np.tril(np.ones((len(idx), len(idx)), dtype=bool))
        Se = np.exp(r)[:, None] * S
        P = s * np.where(mask, Qt @ Kt.T, 0.0)
        o[idx] = P @ v[idx] + s * (Qt @ Se)
        S = np.exp(B - r)[:, None] * (Se + Kt.T @ v[idx])
    return o, S


def gated_backward(q, k, v, do, l, s, S0, dF, C, reverse):
    chunks = _chunks(q.shape[0], C, reverse)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    S = S0.copy()
    for idx in chunks:                                   # dq~: forward order
        Qt, Kt, b, B, r = _rescale(q[idx], k[idx], l[idx])
        mask = np.tril(np.ones((len(idx), len(idx)), dtype=bool))
        Se = np.exp(r)[:, None] * S
        DO, V = do[idx], v[idx]
        dqt = s * (DO @ Se.T + np.where(mask, DO @ V.T, 0.0) @ Kt)
        dq[idx] = dqt * np.exp(b - r)
        S = np.exp(B - r)[:, None] * (Se + Kt.T @ V)
    F = S
    H = dF.copy()
    for idx in reversed(chunks):                         # dv, dk~: against it
        Qt, Kt, b, B, r = _rescale(q[idx], k[idx], l[idx])
        mask = np.tril(np.ones((len(idx), len(idx)), dtype=bool))
        DO, V = do[idx], v[idx]
        Hh = np.exp(B - r)[:, None] * H
        A = s * np.where(mask, Qt @ Kt.T, 0.0)
        Bm = s * np.where(mask, DO @ V.T, 0.0)
        dv[idx] = A.T @ DO + Kt @ Hh
        dk[idx] = (Bm.T @ Qt + V @ Hh.T) * np.exp(r - b)
        H = np.exp(r)[:, None] * (s * Qt.T @ DO + Hh)
    order = np.concatenate(chunks) if chunks else np.arange(0)
    term = q * dq - k * dk
    if len(order):
        term[order[-1]] += (F * dF).sum(-1)
    dg = np.zeros_like(q)
    dg[order] = np.cumsum(term[order][::-1], axis=0)[::-1]
    return dq, dk, dv, dg, H, F


def _run(x, C, reverse):
    q, k, v, do, g = (x[n].numpy() for n in ("q", "k", "v", "do", "g"))
    gg = x["g_gamma"].numpy()
    init, dfin = x["initial_state"].numpy(), x["d_final_state"].numpy()
    cu = x["cu_seqlens"]
    spans = ([(b, 0, q.shape[1], b) for b in range(q.shape[0])] if cu is None else
             [(0, int(cu[n]), int(cu[n + 1]), n) for n in range(len(cu) - 1)])
    out = {n: np.zeros_like(t) for n, t in
           (("o", v), ("dq", q), ("dk", k), ("dv", v), ("dg", q))}
    fin, dinit = np.zeros_like(init), np.zeros_like(init)
    for row, a, b, n in spans:
        for h in range(q.shape[2]):
            sl = (row, slice(a, b), h)
            l = gg[h] + g[sl]
            o, S = gated_forward(q[sl], k[sl], v[sl], l, x["scale"], init[n, h], C, reverse)
            dq, dk, dv, dg, H, F = gated_backward(q[sl], k[sl], v[sl], do[sl], l, x["scale"],
                                                  init[n, h], dfin[n, h], C, reverse)
            assert np.allclose(F, S, rtol=1e-12, atol=0)
            out["o"][sl], out["dq"][sl], out["dk"][sl], out["dv"][sl], out["dg"][sl] = \
                o, dq, dk, dv, dg
            fin[n, h], dinit[n, h] = S, H
    out.update(final_state=fin, d_initial_state=dinit)
    return out


def _oracle(x, reverse):
    args = (x["q"], x["k"], x["v"], x["g"], x["g_gamma"], x["scale"])
    o, fin = oracle.gla_forward(*args, x["initial_state"], reverse, x["cu_seqlens"])
    dq, dk, dv, dg, dinit = oracle.gla_backward(*args, x["do"], x["initial_state"],
                                                x["d_final_state"], reverse, x["cu_seqlens"])
    return dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, dg=dg, d_initial_state=dinit)


def _inputs(seed, B, T, H, d, e, g_lo, g_hi, nseq):
    x = W.random_small(seed, B, T, H, d, e, g_lo=-0.5, g_hi=0.0)
    gen = torch.Generator().manual_seed(seed + 100)
    x["g"] = g_lo + (g_hi - g_lo) * torch.rand((B, T, H, d), generator=gen, dtype=torch.float64)
    x["initial_state"] = torch.randn((nseq, H, d, e), generator=gen, dtype=torch.float64)
    x["d_final_state"] = torch.randn((nseq, H, d, e), generator=gen, dtype=torch.float64)
    return x


def _check(got, ref, tol=1e-9):
    for name, r in ref.items():
        r = np.asarray(r, dtype=np.float64)
        err = np.max(np.abs(got[name] - r)) / max(np.max(np.abs(r)), 1e-300)
        assert err <= tol, (name, err)


@pytest.mark.parametrize("C", [1, 5, 16])
@pytest.mark.parametrize("reverse", [False, True])
def test_gated_chunked_form_equals_the_recurrence(C, reverse):
    x = _inputs(3, 2, 29, 2, 4, 3, -1.0, 0.0, 2)
    x["scale"], x["cu_seqlens"] = 0.8, None
    _check(_run(x, C, reverse), _oracle(x, reverse))


@pytest.mark.parametrize("reverse", [False, True])
def test_gated_chunked_form_packed_with_the_reference_clamped(reverse):
    # strong gates: a 16-token chunk's log-decay reaches about -150, so the
    # midrange of b drops below -72 and r is clamped there
    x = _inputs(7, 1, 40, 2, 3, 4, -10.0, -9.0, 4)
    x["scale"], x["cu_seqlens"] = 0.6, [0, 7, 7, 26, 40]
    l = x["g_gamma"][0].item() + x["g"][0, 7:23, 0].numpy()
    assert (_rescale(l, l, l)[4] == -LIM).all()
    _check(_run(x, 16, reverse), _oracle(x, reverse))
