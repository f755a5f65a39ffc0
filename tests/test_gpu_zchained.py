"""Calls chained on one stream with no host synchronisation between them, each
reading what the one before it wrote: the first forward's output becomes the
second forward's values and the backward's values, its final state the second
forward's initial state, and the second forward's output the backward's
upstream gradient.  The tensor-core sweeps are launched as programmatic
dependents of the stream's previous kernel, so here five of them in a row
(b2 h4 n700 d=e=128 bf16: two forward launches, then la_bwd's dq, dv and dk)
each read data the previous one produced.  The oracle runs the same chain on
its own results, rounded to bf16 / fp32 where the GPU chain stores them."""
import pytest
import torch

import linear_attention_head_gb300 as la
import oracle
import workloads as W
from parity import TOL, compare

pytestmark = pytest.mark.gpu


def test_chained_calls_read_the_previous_calls_outputs():
    B, T, H, D = 2, 700, 4, 128
    w = W.Workload("chain", B, T, H, D, D, torch.bfloat16, W.alibi_g_gamma(H), D ** -0.5)
    x = W.make_inputs(w, seed=23)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    g = x["g_gamma"].cuda()
    o1, f1 = la.la_fwd(q, k, v, g, w.scale)
    o2, f2 = la.la_fwd(q, k, o1, g, w.scale, f1)
    dq, dk, dv, dinit = la.la_bwd(q, k, o1, o2, g, w.scale, f1)
    torch.cuda.synchronize()
    la.get_device_error()

    r1, rf1 = oracle.forward(x["q"], x["k"], x["v"], x["g_gamma"], w.scale)
    o1r = torch.as_tensor(r1).to(torch.bfloat16)
    f1r = torch.as_tensor(rf1).to(torch.float32)
    r2, rf2 = oracle.forward(x["q"], x["k"], o1r, x["g_gamma"], w.scale, f1r)
    o2r = torch.as_tensor(r2).to(torch.bfloat16)
    rq, rk, rv, rinit = oracle.backward(x["q"], x["k"], o1r, x["g_gamma"], w.scale, o2r, f1r)

    tol = TOL[torch.bfloat16]
    compare(dict(o=o1.cpu(), final_state=f1.cpu()), dict(o=r1, final_state=rf1), tol,
            label="first forward")
    compare(dict(o=o2.cpu(), final_state=f2.cpu(), dq=dq.cpu(), dk=dk.cpu(), dv=dv.cpu(),
                 d_initial_state=dinit.cpu()),
            dict(o=r2, final_state=rf2, dq=rq, dk=rk, dv=rv, d_initial_state=rinit), tol,
            label="chained second forward and backward")
