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


def slice_err(x, ref, cu=None, state=False):
    """Max over (sequence, head) slices of max|x-ref| / max|ref|."""
    x, ref = _np(x), _np(ref)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    worst = 0.0
    if state:
        for n in range(ref.shape[0]):
            for h in range(ref.shape[1]):
                a, b = x[n, h], ref[n, h]
                worst = max(worst, np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))
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
            worst = max(worst, np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))
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


def compare(got, ref, tol, cu=None, label=""):
    errs = {}
    for name, r in ref.items():
        errs[name] = slice_err(got[name], r, cu, state=name in ("final_state", "d_initial_state"))
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, "%s: errors above %.1e: %s (all: %s)" % (label, tol, bad, errs)
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
