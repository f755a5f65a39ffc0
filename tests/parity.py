"""Helpers for GPU-vs-oracle parity tests.

Error metric (one reading of "max relative error", which the sources leave
undefined): for every output tensor and every (sequence, head) slice,
max|x - ref| / max|ref|; the test takes the maximum over slices.  Slicing per
head keeps a zero-decay head, whose values grow with the length, from hiding
the error of a fast-decay head.
"""
import numpy as np
import torch

import linear_attention_head_gb300 as la
import oracle

TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}


def _np(t):
    return t.detach().float().cpu().double().numpy() if isinstance(t, torch.Tensor) else t


def _worse(worst, e):
    """Running maximum in which a NaN error (a NaN or inf anywhere in the slice)
    wins: Python's max() would silently keep the previous value."""
    e = float(e)
    return float("inf") if e != e else max(worst, e)


def slice_err(x, ref, cu=None, state=False):
    """Max over (sequence, head) slices of max|x-ref| / max|ref|; inf when any
    slice holds a NaN."""
    x, ref = _np(x), _np(ref)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    worst = 0.0
    if state:
        for n in range(ref.shape[0]):
            for h in range(ref.shape[1]):
                a, b = x[n, h], ref[n, h]
                worst = _worse(worst, np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))
        return worst
    H = ref.shape[2]
    if cu is None:
        segs = [(b, 0, ref.shape[1]) for b in range(ref.shape[0])]
    else:
        cu = [int(c) for c in cu]
        segs = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    for row, s, e in segs:
        if e <= s:
            continue
        for h in range(H):
            a, b = x[row, s:e, h], ref[row, s:e, h]
            worst = _worse(worst, np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))
    return worst


def to_dev(x, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def gpu_run(x, reverse=False, backward=True):
    """x: CPU inputs from workloads.make_inputs; returns CPU results."""
    d = to_dev(x)
    o, fin = la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], d["scale"], d["initial_state"],
                       reverse, x["cu_seqlens"])
    out = dict(o=o, final_state=fin)
    if backward:
        dq, dk, dv, dinit = la.la_bwd(d["q"], d["k"], d["v"], d["do"], d["g_gamma"], d["scale"],
                                      d["initial_state"], d["d_final_state"], reverse,
                                      x["cu_seqlens"])
        out.update(dq=dq, dk=dk, dv=dv, d_initial_state=dinit)
    torch.cuda.synchronize()
    la.get_device_error()
    return {k: v.cpu() for k, v in out.items()}


def oracle_run(x, reverse=False, backward=True, threads=0):
    o, fin = oracle.forward(x["q"], x["k"], x["v"], x["g_gamma"], x["scale"],
                            x["initial_state"], reverse, x["cu_seqlens"], threads=threads)
    out = dict(o=o, final_state=fin)
    if backward:
        dq, dk, dv, dinit = oracle.backward(x["q"], x["k"], x["v"], x["g_gamma"], x["scale"],
                                            x["do"], x["initial_state"], x["d_final_state"],
                                            reverse, x["cu_seqlens"], threads=threads)
        out.update(dq=dq, dk=dk, dv=dv, d_initial_state=dinit)
    return out


def rms_rel(x, ref):
    """Whole-tensor RMS-relative error, reported beside the gated metric."""
    x, ref = _np(x), _np(ref)
    return float(np.sqrt(np.mean((x - ref) ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30))


def compare(got, ref, tol, cu=None, label=""):
    errs = {}
    for name, r in ref.items():
        errs[name] = slice_err(got[name], r, cu, state=name in ("final_state", "d_initial_state"))
    bad = {k: v for k, v in errs.items() if not v <= tol}
    if bad:
        rms = {k: rms_rel(got[k], ref[k]) for k in ref}
        raise AssertionError("%s: errors above %.1e: %s (all: %s; RMS-relative: %s)"
                             % (label, tol, bad, errs, rms))
    return errs


def take_heads(x, heads, rows=None):
    """Restrict CPU inputs to some heads (and batch rows) so the oracle can run on a
    sample of a full-size workload; results compare to the same slice of the GPU run."""
    hs = list(heads)
    y = dict(x)
    for n in ("q", "k", "v", "do"):
        if y.get(n) is not None:
            t = y[n][:, :, hs]
            if rows is not None:
                t = t[list(rows)]
            y[n] = t.contiguous()
    for n in ("initial_state", "d_final_state"):
        if y.get(n) is not None:
            t = y[n][:, hs]
            if rows is not None:
                t = t[list(rows)]
            y[n] = t.contiguous()
    y["g_gamma"] = x["g_gamma"][hs].contiguous()
    return y


def take_out(got, heads, rows=None):
    hs = list(heads)
    y = {}
    for n, t in got.items():
        if n in ("final_state", "d_initial_state"):
            s = t[:, hs]
        else:
            s = t[:, :, hs]
        if rows is not None:
            s = s[list(rows)]
        y[n] = s
    return y


def dg_condition(x, ref, reverse):
    """Per (sequence, head): the largest running sum, in the order dg sums them
    (from the last processed token back), of |q dq| + |k dk| per channel, plus
    sum_e |F dF| -- the scale of dg's rounding error, whatever dg's own size
    (dg is a sum of differences of rounded products, so cancellation can make
    it small while its error is not)."""
    q, k = (np.asarray(x[n].float().numpy(), dtype=np.float64) for n in ("q", "k"))
    dq, dk = np.asarray(ref["dq"], dtype=np.float64), np.asarray(ref["dk"], dtype=np.float64)
    term = np.abs(q * dq) + np.abs(k * dk)                     # [B, T, H, D]
    fin = np.asarray(ref["final_state"], dtype=np.float64)
    dfin = x.get("d_final_state")
    fdf = (np.abs(fin * np.asarray(dfin.numpy(), dtype=np.float64)).sum(-1)
           if dfin is not None else np.zeros(fin.shape[:3]))  # [N, H, D]
    cu = x["cu_seqlens"]
    spans = ([(0, b, 0, q.shape[1]) for b in range(q.shape[0])] if cu is None else
             [(n, 0, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)])
    cond = {}
    for n, row, a, b in spans:
        seg = term[row, a:b]                                   # [L, H, D]
        order = seg if reverse else seg[::-1]                  # dg sums from the last processed
        run = np.cumsum(order, axis=0) + fdf[n if cu is not None else row][None]
        cond[(n if cu is not None else row)] = run.max(axis=(0, 2)) if b > a else fdf[n].max(-1)
    return cond


def compare_gated(got, ref, x, reverse, tol, label, plain_dg_except=()):
    """Every output by the usual per-slice maximum relative error, dg
    included; dg also relative to dg_condition (its error against the scale of
    the sums it is made of).  Returns (plain, conditioned) for dg, or None.
    plain_dg_except: (sequence, head) slices whose dg is held to the
    conditioned bound alone (near-cancelling sums, where the plain ratio
    measures max|dg|, not the error)."""
    rest = {k: v for k, v in ref.items() if k in got and not (k == "dg" and plain_dg_except)}
    errs = compare({k: got[k] for k in rest}, rest, tol, cu=x["cu_seqlens"], label=label)
    if "dg" not in ref:
        return None
    if plain_dg_except:
        g, r = _np(got["dg"]), _np(ref["dg"])
        cu = x["cu_seqlens"]
        worst = 0.0
        for n in range(len(cu) - 1 if cu is not None else g.shape[0]):
            a, b, row = (int(cu[n]), int(cu[n + 1]), 0) if cu is not None else (0, g.shape[1], n)
            for h in range(g.shape[2]):
                if b > a and (n, h) not in plain_dg_except:
                    rr = r[row, a:b, h]
                    worst = _worse(worst, np.abs(g[row, a:b, h] - rr).max() /
                                   max(np.abs(rr).max(), 1e-30))
        assert worst <= tol, "%s: dg error %.3e above %.1e" % (label, worst, tol)
        errs["dg"] = worst
    cond = dg_condition(x, ref, reverse)
    d = np.abs(np.asarray(got["dg"].double().numpy()) - np.asarray(ref["dg"], dtype=np.float64))
    cu = x["cu_seqlens"]
    worst = 0.0
    for key, c in cond.items():
        if cu is None:
            e = d[key].max(axis=(0, 2))
        else:
            a, b = int(cu[key]), int(cu[key + 1])
            if b == a:
                continue
            e = d[0, a:b].max(axis=(0, 2))
        worst = _worse(worst, (e / np.maximum(c, 1e-30)).max())
    assert worst <= tol, "%s: dg error %.3e of its condition above %.1e" % (label, worst, tol)
    return errs["dg"], worst
