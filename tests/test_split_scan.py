"""The sequence split's algebra on the CPU, with the fp64 oracle as the
per-segment runner: every sequence is cut into segments; a first pass from
zero states gives each segment's own contribution F; a scan in visiting order
(carry <- gamma^L carry + F, starting from the initial state) gives each
segment's entering state and the final state; a second pass from those
states gives the outputs.  The backward scans its G = dL/dS the same way
against the visiting order, starting from d_final_state.  Both must reproduce
the unsplit run, because each segment maps its entering state affinely."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _seg_bounds(L, seg):
    return [(a, min(L, a + seg)) for a in range(0, L, seg)]


def _split_run(x, seg, reverse):
    q, k, v, do = (x[n] for n in ("q", "k", "v", "do"))
    g, s = x["g_gamma"], x["scale"]
    S0, dF = x["initial_state"], x["d_final_state"]
    B, T, H, d = q.shape
    e = v.shape[3]
    gamma = torch.exp(g.double())[None, :, None, None]
    segs = _seg_bounds(T, seg)
    visit = segs[::-1] if reverse else segs
    part = lambda t, a, b: t[:, a:b].contiguous()
    zero = torch.zeros((B, H, d, e), dtype=torch.float64)
    # pass 1: each segment from zero states (forward state, backward gradient)
    F = {}
    Gc = {}
    for a, b in segs:
        _, F[a] = oracle.forward(part(q, a, b), part(k, a, b), part(v, a, b), g, s, None,
                                 reverse)
        *_, Gc[a] = oracle.backward(part(q, a, b), part(k, a, b), part(v, a, b), g, s,
                                    part(do, a, b), zero, zero, reverse)
    # scans
    Win, carry = {}, S0.double()
    for a, b in visit:
        Win[a] = carry
        carry = gamma ** (b - a) * carry + torch.as_tensor(F[a])
    final = carry
    Wout, carry = {}, dF.double()
    for a, b in visit[::-1]:
        Wout[a] = carry
        carry = gamma ** (b - a) * carry + torch.as_tensor(Gc[a])
    dinit = carry
    # pass 2
    o = np.zeros((B, T, H, e))
    dq, dk, dv = np.zeros((B, T, H, d)), np.zeros((B, T, H, d)), np.zeros((B, T, H, e))
    for a, b in segs:
        o[:, a:b], _ = oracle.forward(part(q, a, b), part(k, a, b), part(v, a, b), g, s,
                                      Win[a], reverse)
        dq[:, a:b], dk[:, a:b], dv[:, a:b], _ = oracle.backward(
            part(q, a, b), part(k, a, b), part(v, a, b), g, s, part(do, a, b), Win[a],
            Wout[a], reverse)
    return dict(o=o, final_state=final.numpy(), dq=dq, dk=dk, dv=dv,
                d_initial_state=dinit.numpy())


@pytest.mark.parametrize("seg", [1, 7, 16])
@pytest.mark.parametrize("reverse", [False, True])
def test_split_passes_around_a_state_scan_equal_the_unsplit_run(seg, reverse):
    x = W.random_small(11, 2, 45, 3, 4, 5, g_lo=-0.8, g_hi=0.0)
    x["g_gamma"][1] = 0.0
    gen = torch.Generator().manual_seed(12)
    x["initial_state"] = torch.randn((2, 3, 4, 5), generator=gen, dtype=torch.float64)
    x["d_final_state"] = torch.randn((2, 3, 4, 5), generator=gen, dtype=torch.float64)
    x["scale"] = 0.9
    got = _split_run(x, seg, reverse)
    o, fin = oracle.forward(x["q"], x["k"], x["v"], x["g_gamma"], x["scale"],
                            x["initial_state"], reverse)
    dq, dk, dv, dinit = oracle.backward(x["q"], x["k"], x["v"], x["g_gamma"], x["scale"],
                                        x["do"], x["initial_state"], x["d_final_state"],
                                        reverse)
    ref = dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, d_initial_state=dinit)
    for name, r in ref.items():
        r = np.asarray(r)
        err = np.max(np.abs(got[name] - r)) / np.max(np.abs(r))
        assert err <= 1e-12, (name, err)


def _gated_split_forward(x, seg, reverse, gates_in_decay=True):
    """The gated forward split: per segment, its state from zero (oracle) and
    its log-decay per key channel (len * g_gamma + the sum of its gates); the
    scan carry <- diag(exp(lam)) carry + F in visiting order; pass 2 from the
    scanned states.  gates_in_decay=False plants a mistake: the scan's decay
    without the gates' sum."""
    q, k, v, gt = (x[n] for n in ("q", "k", "v", "g"))
    gg, s, S0 = x["g_gamma"], x["scale"], x["initial_state"]
    T = q.shape[1]
    segs = _seg_bounds(T, seg)
    visit = segs[::-1] if reverse else segs
    part = lambda t, a, b: t[:, a:b].contiguous()
    F, lam = {}, {}
    for a, b in segs:
        _, F[a] = oracle.gla_forward(part(q, a, b), part(k, a, b), part(v, a, b),
                                     part(gt, a, b), gg, s, None, reverse)
        lam[a] = (b - a) * gg.double()[None, :, None] + \
            (gt[:, a:b].double().sum(1) if gates_in_decay else 0.0)   # [B, H, d]
    Win, carry = {}, S0.double()
    for a, b in visit:
        Win[a] = carry
        carry = torch.exp(lam[a])[..., None] * carry + torch.as_tensor(F[a])
    o = np.zeros(q.shape[:3] + v.shape[3:])
    for a, b in segs:
        o[:, a:b], _ = oracle.gla_forward(part(q, a, b), part(k, a, b), part(v, a, b),
                                          part(gt, a, b), gg, s, Win[a], reverse)
    return o, carry.numpy()


@pytest.mark.parametrize("seg", [1, 6, 16])
@pytest.mark.parametrize("reverse", [False, True])
def test_gated_split_scans_with_per_channel_decays(seg, reverse):
    # the gated form's segment decay is a diagonal (one factor per key
    # channel, the state's rows), so the scan stays elementwise
    x = W.random_small(13, 2, 40, 3, 4, 5, g_lo=-0.5, g_hi=0.0)
    gen = torch.Generator().manual_seed(14)
    x["g"] = -0.6 * torch.rand(x["q"].shape, generator=gen, dtype=torch.float64)
    x["initial_state"] = torch.randn((2, 3, 4, 5), generator=gen, dtype=torch.float64)
    x["scale"] = 0.8
    o, fin = _gated_split_forward(x, seg, reverse)
    ro, rfin = oracle.gla_forward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"], x["scale"],
                                  x["initial_state"], reverse)
    assert np.abs(o - np.asarray(ro)).max() <= 1e-12 * max(1.0, np.abs(ro).max())
    assert np.abs(fin - np.asarray(rfin)).max() <= 1e-12 * max(1.0, np.abs(rfin).max())
    # the scan with the head's decay gamma^L alone (the gates left out) fails
    if len(_seg_bounds(40, seg)) > 1:
        o_bad, fin_bad = _gated_split_forward(x, seg, reverse, gates_in_decay=False)
        # (the older state has mostly decayed over a segment, so the outputs
        # move by 1e-3 of their maximum or less: far above the 1e-12 match)
        assert np.abs(o_bad - np.asarray(ro)).max() > 1e-6 * np.abs(ro).max()
        assert np.abs(fin_bad - np.asarray(rfin)).max() > 1e-6 * np.abs(rfin).max()


def _gated_split_backward(x, seg, reverse, g_decay_on_rows=True):
    """The gated backward split through the oracle: pass 1 gives each
    segment's state from zero (forward) and its dL/dS at entry from a zero
    gradient at its end (backward); the scans carry S forward and G against
    the visiting order, both with the segment's per-key-channel decay
    diag(exp(lam)) on the key rows; pass 2 runs each segment's backward from
    its entering S and the G that arrives from the segments after it.
    g_decay_on_rows=False plants a mistake: G's decay on the value columns."""
    q, k, v, gt, do = (x[n] for n in ("q", "k", "v", "g", "do"))
    gg, s = x["g_gamma"], x["scale"]
    S0, dF = x["initial_state"], x["d_final_state"]
    B, T, H, d = q.shape
    e = v.shape[3]
    segs = _seg_bounds(T, seg)
    visit = segs[::-1] if reverse else segs
    part = lambda t, a, b: t[:, a:b].contiguous()
    zero = torch.zeros((B, H, d, e), dtype=torch.float64)
    F, Gc, lam = {}, {}, {}
    for a, b in segs:
        args = (part(q, a, b), part(k, a, b), part(v, a, b), part(gt, a, b), gg, s)
        _, F[a] = oracle.gla_forward(*args, None, reverse)
        *_, Gc[a] = oracle.gla_backward(*args, part(do, a, b), zero, zero, reverse)
        lam[a] = torch.exp((b - a) * gg.double()[None, :, None] + gt[:, a:b].double().sum(1))
    Win, carry = {}, S0.double()
    for a, b in visit:
        Win[a] = carry
        carry = lam[a][..., None] * carry + torch.as_tensor(F[a])
    Wout, carry = {}, dF.double()
    for a, b in visit[::-1]:
        Wout[a] = carry
        dec = lam[a][..., None] if g_decay_on_rows else lam[a][..., None, :e]
        carry = dec * carry + torch.as_tensor(Gc[a])
    dinit = carry
    out = {n: np.zeros(t.shape) for n, t in (("dq", q), ("dk", k), ("dv", v), ("dg", gt))}
    for a, b in segs:
        dq, dk, dv, dg, _ = oracle.gla_backward(part(q, a, b), part(k, a, b), part(v, a, b),
                                                part(gt, a, b), gg, s, part(do, a, b), Win[a],
                                                Wout[a], reverse)
        for n, t in (("dq", dq), ("dk", dk), ("dv", dv), ("dg", dg)):
            out[n][:, a:b] = np.asarray(t)
    out["d_initial_state"] = dinit.numpy()
    return out


@pytest.mark.parametrize("seg", [1, 6, 16])
@pytest.mark.parametrize("reverse", [False, True])
def test_gated_split_backward_scans_with_per_channel_decays(seg, reverse):
    # dq, dk, dv, dg and d_initial_state of the whole sequence from the
    # segments' backward runs around the two scans (per-key-channel decays
    # on the key rows of S and of G = dL/dS)
    x = W.random_small(17, 2, 40, 3, 4, 4, g_lo=-0.5, g_hi=0.0)
    gen = torch.Generator().manual_seed(18)
    x["g"] = -0.6 * torch.rand(x["q"].shape, generator=gen, dtype=torch.float64)
    x["initial_state"] = torch.randn((2, 3, 4, 4), generator=gen, dtype=torch.float64)
    x["d_final_state"] = torch.randn((2, 3, 4, 4), generator=gen, dtype=torch.float64)
    x["scale"] = 0.8
    got = _gated_split_backward(x, seg, reverse)
    dq, dk, dv, dg, dinit = oracle.gla_backward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"],
                                                x["scale"], x["do"], x["initial_state"],
                                                x["d_final_state"], reverse)
    ref = dict(dq=dq, dk=dk, dv=dv, dg=dg, d_initial_state=dinit)
    for name, r in ref.items():
        r = np.asarray(r)
        assert np.abs(got[name] - r).max() <= 1e-11 * max(1.0, np.abs(r).max()), name
    # G's decay applied to its value columns instead of its key rows fails
    if len(_seg_bounds(40, seg)) > 1:
        bad = _gated_split_backward(x, seg, reverse, g_decay_on_rows=False)
        assert np.abs(bad["dk"] - np.asarray(dk)).max() > 1e-6 * np.abs(np.asarray(dk)).max()
