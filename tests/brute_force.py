"""Brute-force quadratic (attention-matrix) form of decayed causal linear
attention, used only to pin the recurrent fp64 oracle.

Unrolling the recurrence S_t = gamma S_{t-1} + outer(k_t, v_t) (ejkernel
`recurrent` docstring, its state-update formula) from S_0 gives, for the token at
processing position p(t) (p(t) = t, or L-1-t when reversed):

  o_t   = s * sum_{u: p(u) <= p(t)} gamma^(p(t)-p(u)) (q_t . k_u) v_u
          + s * gamma^(p(t)+1) * q_t^T S_0
  final = gamma^L S_0 + sum_u gamma^(L-1-p(u)) outer(k_u, v_u)

and, for the loss sum(o*do) + sum(final*dF),

  dq_t  = s * sum_{p(u) <= p(t)} gamma^(p(t)-p(u)) (do_t . v_u) k_u + s gamma^(p(t)+1) S_0 do_t
  dk_u  = s * sum_{p(t) >= p(u)} gamma^(p(t)-p(u)) (do_t . v_u) q_t + gamma^(L-1-p(u)) dF v_u
  dv_u  = s * sum_{p(t) >= p(u)} gamma^(p(t)-p(u)) (q_t . k_u) do_t + gamma^(L-1-p(u)) dF^T k_u
  dS_0  = s * sum_t gamma^(p(t)+1) outer(q_t, do_t) + gamma^L dF

Everything here is an explicit double loop over (t, u) pairs in float64 (numpy
only for the dot products), so it is O(L^2) and only meant for tiny inputs.
"""
import numpy as np


def _single(q, k, v, g, s, S0, reverse, do=None, dF=None):
    """One (sequence, head): q,k [L,d], v,do [L,e], S0,dF [d,e] or None."""
    L, d = q.shape
    e = v.shape[1]
    gam = np.exp(g)
    pos = np.arange(L)[::-1] if reverse else np.arange(L)
    S0 = np.zeros((d, e)) if S0 is None else S0
    dF = np.zeros((d, e)) if dF is None else dF
    o = np.zeros((L, e))
    fin = gam ** L * S0
    for t in range(L):
        for u in range(L):
            if pos[u] <= pos[t]:
                o[t] += s * gam ** (pos[t] - pos[u]) * np.dot(q[t], k[u]) * v[u]
        o[t] += s * gam ** (pos[t] + 1) * (q[t] @ S0)
    for u in range(L):
        fin = fin + gam ** (L - 1 - pos[u]) * np.outer(k[u], v[u])
    if do is None:
        return o, fin
    dq = np.zeros((L, d))
    dk = np.zeros((L, d))
    dv = np.zeros((L, e))
    dS0 = gam ** L * dF
    for t in range(L):
        for u in range(L):
            if pos[u] <= pos[t]:
                w = s * gam ** (pos[t] - pos[u])
                dq[t] += w * np.dot(do[t], v[u]) * k[u]
                dk[u] += w * np.dot(do[t], v[u]) * q[t]
                dv[u] += w * np.dot(q[t], k[u]) * do[t]
        dq[t] += s * gam ** (pos[t] + 1) * (S0 @ do[t])
        dS0 = dS0 + s * gam ** (pos[t] + 1) * np.outer(q[t], do[t])
    for u in range(L):
        dk[u] += gam ** (L - 1 - pos[u]) * (dF @ v[u])
        dv[u] += gam ** (L - 1 - pos[u]) * (dF.T @ k[u])
    return o, fin, dq, dk, dv, dS0


def brute(q, k, v, g_gamma, scale, initial_state=None, reverse=False, cu_seqlens=None,
          do=None, d_final_state=None):
    """Same conventions as oracle.forward / oracle.backward, all float64 numpy.
    Returns (o, final) or (o, final, dq, dk, dv, d_initial_state)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, T, H, d = q.shape
    e = v.shape[3]
    g = np.broadcast_to(np.asarray(g_gamma, dtype=np.float64), (H,))
    if cu_seqlens is None:
        segs = [(b, 0, T) for b in range(B)]
    else:
        cu = [int(c) for c in cu_seqlens]
        segs = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    N = len(segs)
    o = np.zeros((B, T, H, e))
    fin = np.zeros((N, H, d, e))
    grads = do is not None
    if grads:
        do = np.asarray(do, dtype=np.float64)
        dq = np.zeros_like(q)
        dk = np.zeros_like(k)
        dv = np.zeros_like(v)
        dS0 = np.zeros((N, H, d, e))
    for n, (row, a, b) in enumerate(segs):
        for h in range(H):
            S0 = None if initial_state is None else np.asarray(initial_state, np.float64)[n, h]
            dF = None if d_final_state is None else np.asarray(d_final_state, np.float64)[n, h]
            res = _single(q[row, a:b, h], k[row, a:b, h], v[row, a:b, h], g[h], scale, S0,
                          reverse, None if not grads else do[row, a:b, h], dF)
            o[row, a:b, h] = res[0]
            fin[n, h] = res[1]
            if grads:
                dq[row, a:b, h], dk[row, a:b, h], dv[row, a:b, h], dS0[n, h] = res[2:]
    if grads:
        return o, fin, dq, dk, dv, dS0
    return o, fin
