"""Grouped key/value heads on the CPU: query head h reads key/value head
h // G, and the gradient of a shared key or value is the sum of its query
heads' gradients.  Pinned by finite differences of the loss through the
oracle run on the repeated heads (a perturbation of a shared element moves
every copy), not by the summation itself."""
import numpy as np
import torch

import oracle
import workloads as W


def _loss(q, k_kv, v_kv, g, s, do, G):
    k = k_kv.repeat_interleave(G, dim=2)
    v = v_kv.repeat_interleave(G, dim=2)
    o, _ = oracle.forward(q, k, v, g, s)
    return float((np.asarray(o) * do.numpy()).sum())


def test_shared_head_gradient_is_the_sum_over_its_group():
    B, T, H, Hkv, d, e = 1, 13, 4, 2, 3, 2
    G = H // Hkv
    x = W.random_small(21, B, T, H, d, e, g_lo=-0.6, g_hi=0.0)
    q, do, g = x["q"], x["do"], x["g_gamma"]
    k_kv, v_kv = x["k"][:, :, :Hkv].clone(), x["v"][:, :, :Hkv].clone()
    s = 0.7
    k, v = k_kv.repeat_interleave(G, dim=2), v_kv.repeat_interleave(G, dim=2)
    _, dk, dv, _ = oracle.backward(q, k, v, g, s, do)
    dk_kv = np.asarray(dk).reshape(B, T, Hkv, G, d).sum(3)
    dv_kv = np.asarray(dv).reshape(B, T, Hkv, G, e).sum(3)
    eps = 1e-6
    for (t, hk, c) in [(0, 0, 1), (6, 1, 2), (12, 1, 0)]:
        kp, km = k_kv.clone(), k_kv.clone()
        kp[0, t, hk, c] += eps
        km[0, t, hk, c] -= eps
        fd = (_loss(q, kp, v_kv, g, s, do, G) - _loss(q, km, v_kv, g, s, do, G)) / (2 * eps)
        assert abs(fd - dk_kv[0, t, hk, c]) <= 1e-7 * max(1.0, abs(fd))
    for (t, hk, c) in [(2, 0, 0), (9, 1, 1)]:
        vp, vm = v_kv.clone(), v_kv.clone()
        vp[0, t, hk, c] += eps
        vm[0, t, hk, c] -= eps
        fd = (_loss(q, k_kv, vp, g, s, do, G) - _loss(q, k_kv, vm, g, s, do, G)) / (2 * eps)
        assert abs(fd - dv_kv[0, t, hk, c]) <= 1e-7 * max(1.0, abs(fd))
    # a single query head's gradient alone is not the shared gradient
    assert not np.allclose(np.asarray(dk)[:, :, 0], dk_kv[:, :, 0])


def _gated_loss(q, k_kv, v_kv, gate, gg, s, do, init, dfin, G, reverse):
    k = k_kv.repeat_interleave(G, dim=2)
    v = v_kv.repeat_interleave(G, dim=2)
    o, fin = oracle.gla_forward(q, k, v, gate, gg, s, init, reverse)
    return float((np.asarray(o) * do.numpy()).sum() + (np.asarray(fin) * dfin.numpy()).sum())


def test_gated_shared_head_gradient_is_the_sum_over_its_group():
    # the gated form with grouped key/value heads: the gate and the state are
    # the query head's, keys and values are shared; dk and dv of a shared head
    # are the group sums, dq and dg those of the repeated-head problem
    B, T, H, Hkv, d, e = 1, 11, 6, 2, 3, 2
    G = H // Hkv
    x = W.random_small(33, B, T, H, d, e, g_lo=-0.4, g_hi=0.0)
    q, do, gg = x["q"], x["do"], x["g_gamma"]
    k_kv, v_kv = x["k"][:, :, :Hkv].clone(), x["v"][:, :, :Hkv].clone()
    gen = torch.Generator().manual_seed(5)
    gate = -0.5 * torch.rand(q.shape, generator=gen, dtype=torch.float64)
    init = torch.randn((B, H, d, e), generator=gen, dtype=torch.float64)
    dfin = torch.randn((B, H, d, e), generator=gen, dtype=torch.float64)
    s = 0.6
    for reverse in (False, True):
        k, v = k_kv.repeat_interleave(G, dim=2), v_kv.repeat_interleave(G, dim=2)
        dq, dk, dv, dg, _ = oracle.gla_backward(q, k, v, gate, gg, s, do, init, dfin, reverse)
        dk_kv = np.asarray(dk).reshape(B, T, Hkv, G, d).sum(3)
        dv_kv = np.asarray(dv).reshape(B, T, Hkv, G, e).sum(3)
        L = lambda kk=k_kv, vv=v_kv, gt=gate: _gated_loss(q, kk, vv, gt, gg, s, do, init, dfin,
                                                         G, reverse)
        eps = 1e-6
        for (t, hk, c) in [(0, 0, 1), (5, 1, 2), (10, 1, 0)]:
            kp, km = k_kv.clone(), k_kv.clone()
            kp[0, t, hk, c] += eps
            km[0, t, hk, c] -= eps
            fd = (L(kk=kp) - L(kk=km)) / (2 * eps)
            assert abs(fd - dk_kv[0, t, hk, c]) <= 1e-7 * max(1.0, abs(fd))
        for (t, hk, c) in [(3, 0, 0), (8, 1, 1)]:
            vp, vm = v_kv.clone(), v_kv.clone()
            vp[0, t, hk, c] += eps
            vm[0, t, hk, c] -= eps
            fd = (L(vv=vp) - L(vv=vm)) / (2 * eps)
            assert abs(fd - dv_kv[0, t, hk, c]) <= 1e-7 * max(1.0, abs(fd))
        for (t, h, c) in [(2, 1, 0), (7, 4, 2)]:
            gp, gm = gate.clone(), gate.clone()
            gp[0, t, h, c] += eps
            gm[0, t, h, c] -= eps
            fd = (L(gt=gp) - L(gt=gm)) / (2 * eps)
            assert abs(fd - np.asarray(dg)[0, t, h, c]) <= 1e-7 * max(1.0, abs(fd))
        # the group's query heads see different gates: their parts differ
        assert not np.allclose(np.asarray(dk)[:, :, 0], np.asarray(dk)[:, :, 1])
