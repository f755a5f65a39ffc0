"""CUDA-graph capture of dense calls.

A call without cu_seqlens whose sequence split does not engage enqueues only
kernels and memsets on the caller's stream (tensor maps are encoded on the
host and travel as kernel parameters), so it can be captured once and
replayed: the launch-bound short calls (decode) pay one graph launch instead
of one host call per kernel.  Captured here: la_fwd + la_bwd on the
tensor-core, decode and CUDA-core paths, and la_gla_fwd + la_gla_bwd on the
chunked gated path.  Replays after new inputs are copied into the captured
buffers equal eager calls on the same inputs bit for bit, and the oracle to
the parity tolerance.  (Packed calls and split calls copy schedule and
segment tables from pageable host memory: they are not captured.)
"""
import math

import pytest
import torch

import linear_attention_head_gb300 as la
import oracle
import workloads as W
from linear_attention_head_gb300 import _native as N
from parity import TOL, compare

pytestmark = pytest.mark.gpu

CASES = {
    "tensor_core": (2, 300, 4, 128, 128, torch.bfloat16),
    "decode": (4, 16, 8, 128, 128, torch.bfloat16),
    "cuda_core": (2, 200, 2, 64, 64, torch.float32),
    "gated": (2, 300, 3, 128, 128, torch.bfloat16),
}


def _draw(B, T, H, D, E, dtype, seed):
    w = W.Workload("graph", B, T, H, D, E, dtype, W.alibi_g_gamma(H), 1.0 / math.sqrt(D),
                   init_std=0.2, dfinal_std=0.2)
    x = W.make_inputs(w, seed=seed)
    x["g"] = -0.3 * torch.rand(x["q"].shape, generator=torch.Generator().manual_seed(seed + 7))
    return x


def _step(kind, d):
    """One forward + backward through the Python binding on device tensors d."""
    if kind == "gated":
        o, fin = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], d["scale"],
                            d["initial_state"])
        dq, dk, dv, dg, dinit = la.gla_bwd(d["q"], d["k"], d["v"], d["do"], d["g"],
                                           d["g_gamma"], d["scale"], d["initial_state"],
                                           d["d_final_state"])
        return dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, dg=dg, d_initial_state=dinit)
    o, fin = la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], d["scale"], d["initial_state"])
    dq, dk, dv, dinit = la.la_bwd(d["q"], d["k"], d["v"], d["do"], d["g_gamma"], d["scale"],
                                  d["initial_state"], d["d_final_state"])
    return dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, d_initial_state=dinit)


def _oracle(kind, x):
    if kind == "gated":
        o, fin = oracle.gla_forward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"], x["scale"],
                                    x["initial_state"])
        dq, dk, dv, dg, dinit = oracle.gla_backward(x["q"], x["k"], x["v"], x["g"],
                                                    x["g_gamma"], x["scale"], x["do"],
                                                    x["initial_state"], x["d_final_state"])
        return dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, dg=dg, d_initial_state=dinit)
    o, fin = oracle.forward(x["q"], x["k"], x["v"], x["g_gamma"], x["scale"], x["initial_state"])
    dq, dk, dv, dinit = oracle.backward(x["q"], x["k"], x["v"], x["g_gamma"], x["scale"],
                                        x["do"], x["initial_state"], x["d_final_state"])
    return dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, d_initial_state=dinit)


NAMES = ("q", "k", "v", "do", "g", "initial_state", "d_final_state", "g_gamma")


@pytest.mark.parametrize("kind", list(CASES))
def test_dense_step_replays_from_a_cuda_graph(kind):
    lib = N.lib()
    assert lib.la_set_sequence_split(0, 0) == N.LA_OK   # no split: nothing copied from the host
    try:
        x0 = _draw(*CASES[kind], seed=0)
        # the captured buffers: every input on the device, g_gamma included
        # (a host tensor would be copied inside the capture)
        d = {n: x0[n].cuda() for n in NAMES}
        d["scale"] = x0["scale"]
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):       # warm-up: first-call set-up outside the capture
            for _ in range(2):
                _step(kind, d)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            out = _step(kind, d)
        launches = lib.la_launch_count()
        for seed in (1, 2):
            x = _draw(*CASES[kind], seed=seed)
            for n in NAMES:
                d[n].copy_(x[n])
            graph.replay()
            torch.cuda.synchronize()
            la.get_device_error()
            got = {k: v.cpu() for k, v in out.items()}
            assert lib.la_launch_count() == launches   # the replay went through no host call
            eager = {k: v.cpu() for k, v in _step(kind, d).items()}
            torch.cuda.synchronize()
            launches = lib.la_launch_count()
            for k in got:
                assert torch.equal(got[k], eager[k]), (kind, seed, k)
            compare(got, _oracle(kind, x), TOL[x["q"].dtype],
                    label="graph %s seed %d" % (kind, seed))
        del graph
    finally:
        lib.la_set_sequence_split(1, 0)
