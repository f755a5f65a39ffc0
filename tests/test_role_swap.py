"""The role swaps by which the library computes every gradient with the two
sweep shapes, checked on the CPU with the oracle playing both shapes:
  dq = the forward sweep on (q, k, v) := (do, v, k) from the transposed
       initial state;
  dv = the backward sweep on (k, q, do), carrying G = dL/dS from d_final_state;
  dk = the same backward sweep on (k, q, do) := (v, do, q), carrying G^T from
       d_final_state^T, whose d_initial_state comes out transposed.
Both directions and packed sequences."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _t(x):
    return x.transpose(-1, -2).contiguous()


@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("packed", [False, True])
def test_gradients_by_role_swap(reverse, packed):
    B, T, H, d, e = (1, 30, 2, 4, 3) if packed else (2, 19, 2, 4, 3)
    cu = [0, 11, 11, 30] if packed else None
    N = 3 if packed else B
    x = W.random_small(31, B, T, H, d, e, g_lo=-0.9, g_hi=0.0)
    q, k, v, do, g = x["q"], x["k"], x["v"], x["do"], x["g_gamma"]
    gen = torch.Generator().manual_seed(32)
    S0 = torch.randn((N, H, d, e), generator=gen, dtype=torch.float64)
    dF = torch.randn((N, H, d, e), generator=gen, dtype=torch.float64)
    s = 0.8
    dq, dk, dv, dinit = oracle.backward(q, k, v, g, s, do, S0, dF, reverse, cu)
    # dq: forward shape on (do, v, k) from S0^T
    dq_swap, _ = oracle.forward(do, v, k, g, s, _t(S0), reverse, cu)
    # dv: the backward shape's own dv output (roles as given)
    # dk: the backward shape on (v, do, q) with d_final_state^T; its "dv" is dk
    _, _, dk_swap, dinit_t = oracle.backward(do, v, k, g, s, q, _t(S0), _t(dF), reverse, cu)
    for a, b in ((dq_swap, dq), (dk_swap, dk), (_t(torch.as_tensor(dinit_t)), dinit)):
        a, b = np.asarray(a), np.asarray(b)
        assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(b))
    assert np.max(np.abs(np.asarray(dv))) > 0
