"""fp64 CPU oracle for causal linear attention with per-head scalar decay.

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference legs may import this package; the product package
(linear_attention_head_gb300) never does, and this package never imports it.

The arithmetic lives in la_oracle.c (plain C, fp64, token by token): the
recurrence of the ejkernel `recurrent` docstring (its state-update formula),
S_t = exp(g_gamma[h]) * S_{t-1} + outer(k_t, v_t), o_t = scale * q_t^T S_t,
with initial_state, reverse and packed cu_seqlens, and the gradient of
sum(o*do) + sum(final*dfinal) with respect to q, k, v and initial_state
(the `_recurrent_bwd` custom VJP on the same page; g_gamma, scale, reverse and
cu_seqlens are not differentiated).  gla_forward / gla_backward add the
per-key gate g [B,T,H,d] (the page's GLA-style gate, read as a log-decay per
key channel added to g_gamma) and its gradient dg.  This module only marshals
numpy arrays.

Pins: every function here is checked in tests/test_oracle_*.py against a
brute-force quadratic form, closed forms, invariants and finite differences.
"""
import ctypes
import numpy as np

from . import build as _build

_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.la_oracle_fwd.restype = ctypes.c_int
        lib.la_oracle_fwd.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, _ip, _dp, _dp, _dp, _dp, ctypes.c_double, _dp,
            ctypes.c_int, _dp, _dp, ctypes.c_int]
        lib.la_oracle_bwd.restype = ctypes.c_int
        lib.la_oracle_bwd.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, _ip, _dp, _dp, _dp, _dp, ctypes.c_double, _dp,
            ctypes.c_int, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int]
        lib.la_oracle_gla_fwd.restype = ctypes.c_int
        lib.la_oracle_gla_fwd.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, _ip, _dp, _dp, _dp, _dp, _dp, ctypes.c_double, _dp,
            ctypes.c_int, _dp, _dp, ctypes.c_int]
        lib.la_oracle_gla_bwd.restype = ctypes.c_int
        lib.la_oracle_gla_bwd.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, _ip, _dp, _dp, _dp, _dp, _dp, ctypes.c_double, _dp,
            ctypes.c_int, _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int]
        _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):           # a CPU torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, typ=_dp):
    return None if a is None else a.ctypes.data_as(typ)


def _check(q, k, v, cu_seqlens, initial_state):
    if q.ndim != 4 or k.shape != q.shape or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k must be [B,T,H,d] and v [B,T,H,e]")
    B, T, H, d = q.shape
    e = v.shape[3]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        if B != 1:
            raise ValueError("cu_seqlens needs batch 1")
        if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("bad cu_seqlens")
        N = cu.size - 1
    else:
        cu = None
        N = B
    if initial_state is not None and initial_state.shape != (N, H, d, e):
        raise ValueError("initial_state must be [N,H,d,e]")
    return B, T, H, d, e, N, cu


def forward(q, k, v, g_gamma, scale, initial_state=None, reverse=False,
            cu_seqlens=None, threads=0):
    """Returns (o [B,T,H,e], final_state [N,H,d,e]) in float64."""
    q, k, v, g, init = map(_f64, (q, k, v, g_gamma, initial_state))
    B, T, H, d, e, N, cu = _check(q, k, v, cu_seqlens, init)
    g = np.ascontiguousarray(np.broadcast_to(g, (H,)))
    o = np.zeros((B, T, H, e))
    fin = np.zeros((N, H, d, e))
    rc = _load().la_oracle_fwd(B, T, H, d, e, N, _ptr(cu, _ip), _ptr(q), _ptr(k), _ptr(v),
                               _ptr(g), float(scale), _ptr(init), int(bool(reverse)),
                               _ptr(o), _ptr(fin), int(threads))
    if rc:
        raise RuntimeError("la_oracle_fwd failed (%d)" % rc)
    return o, fin


def backward(q, k, v, g_gamma, scale, dout, initial_state=None, d_final_state=None,
             reverse=False, cu_seqlens=None, threads=0):
    """Returns (dq, dk [B,T,H,d], dv [B,T,H,e], d_initial_state [N,H,d,e])."""
    q, k, v, g, init, do, dfin = map(_f64, (q, k, v, g_gamma, initial_state, dout,
                                            d_final_state))
    B, T, H, d, e, N, cu = _check(q, k, v, cu_seqlens, init)
    if do.shape != v.shape:
        raise ValueError("dout must match v")
    if dfin is not None and dfin.shape != (N, H, d, e):
        raise ValueError("d_final_state must be [N,H,d,e]")
    g = np.ascontiguousarray(np.broadcast_to(g, (H,)))
    dq = np.zeros((B, T, H, d))
    dk = np.zeros((B, T, H, d))
    dv = np.zeros((B, T, H, e))
    dinit = np.zeros((N, H, d, e))
    rc = _load().la_oracle_bwd(B, T, H, d, e, N, _ptr(cu, _ip), _ptr(q), _ptr(k), _ptr(v),
                               _ptr(g), float(scale), _ptr(init), int(bool(reverse)),
                               _ptr(do), _ptr(dfin), _ptr(dq), _ptr(dk), _ptr(dv),
                               _ptr(dinit), int(threads))
    if rc:
        raise RuntimeError("la_oracle_bwd failed (%d)" % rc)
    return dq, dk, dv, dinit


def gla_forward(q, k, v, g, g_gamma, scale, initial_state=None, reverse=False,
                cu_seqlens=None, threads=0):
    """Gated forward, g [B,T,H,d]: returns (o, final_state) in float64."""
    q, k, v, gt, gg, init = map(_f64, (q, k, v, g, g_gamma, initial_state))
    B, T, H, d, e, N, cu = _check(q, k, v, cu_seqlens, init)
    if gt.shape != q.shape:
        raise ValueError("g must have the keys' shape")
    gg = np.ascontiguousarray(np.broadcast_to(gg, (H,)))
    o = np.zeros((B, T, H, e))
    fin = np.zeros((N, H, d, e))
    rc = _load().la_oracle_gla_fwd(B, T, H, d, e, N, _ptr(cu, _ip), _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(gg), _ptr(gt), float(scale), _ptr(init),
                                   int(bool(reverse)), _ptr(o), _ptr(fin), int(threads))
    if rc:
        raise RuntimeError("la_oracle_gla_fwd failed (%d)" % rc)
    return o, fin


def gla_backward(q, k, v, g, g_gamma, scale, dout, initial_state=None, d_final_state=None,
                 reverse=False, cu_seqlens=None, threads=0):
    """Gated backward: returns (dq, dk, dv, dg, d_initial_state) in float64."""
    q, k, v, gt, gg, init, do, dfin = map(_f64, (q, k, v, g, g_gamma, initial_state, dout,
                                                 d_final_state))
    B, T, H, d, e, N, cu = _check(q, k, v, cu_seqlens, init)
    if gt.shape != q.shape or do.shape != v.shape:
        raise ValueError("g must have the keys' shape and dout the values'")
    if dfin is not None and dfin.shape != (N, H, d, e):
        raise ValueError("d_final_state must be [N,H,d,e]")
    gg = np.ascontiguousarray(np.broadcast_to(gg, (H,)))
    dq, dk, dg = np.zeros((B, T, H, d)), np.zeros((B, T, H, d)), np.zeros((B, T, H, d))
    dv = np.zeros((B, T, H, e))
    dinit = np.zeros((N, H, d, e))
    rc = _load().la_oracle_gla_bwd(B, T, H, d, e, N, _ptr(cu, _ip), _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(gg), _ptr(gt), float(scale), _ptr(init),
                                   int(bool(reverse)), _ptr(do), _ptr(dfin), _ptr(dq), _ptr(dk),
                                   _ptr(dv), _ptr(dg), _ptr(dinit), int(threads))
    if rc:
        raise RuntimeError("la_oracle_gla_bwd failed (%d)" % rc)
    return dq, dk, dv, dg, dinit
