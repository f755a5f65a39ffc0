"""Gated forward with the sequence split: few (sequence, head) pairs, long
sequences.

The segments run as packed sequences in two passes around a scan whose
decay is per key channel (exp of the segment's summed log-decays).  Checked
against the oracle (o, final state) in both directions for dense rows, a
dense batch viewed as one row, packed sequences (shorter than a segment,
empty), value width 64, segments whose gates leave the chunked form's range
(token by token in both passes), a gate layout without a one-row view
(unsplit), and a training step through autograd (the backward, which does
not split, recomputes its operands).
"""
import ctypes
import math

import pytest
import torch

import linear_attention_head_gb300 as la
import oracle
import workloads as W
from linear_attention_head_gb300 import _native as N
from parity import TOL, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def short_segments():
    N.check(N.lib().la_set_sequence_split(1, 256))
    yield
    N.check(N.lib().la_set_sequence_split(1, 0))


def _inputs(B, T, H, E, seqlens=None, seed=0):
    w = W.Workload("gla_split", B, T if seqlens is None else sum(seqlens), H, 128, E,
                   torch.bfloat16, W.alibi_g_gamma(H), 1.0 / math.sqrt(128), seqlens=seqlens,
                   init_std=0.2, dfinal_std=0.2)
    x = W.make_inputs(w, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1000)
    x["g"] = -0.3 * torch.rand(x["q"].shape, generator=gen)
    return x


def _fwd_ws_bytes(x, split):
    d = N.LaDims()
    B, T, H, D = x["q"].shape
    E = x["v"].shape[3]
    cu = x["cu_seqlens"]
    d.batch, d.seq_len, d.heads, d.dim_qk, d.dim_v = B, T, H, D, E
    d.num_seqs = 0 if cu is None else len(cu) - 1
    for i in range(3):
        d.qk_strides[i] = x["q"].stride(i)
        d.v_strides[i] = x["v"].stride(i)
    keep = None if cu is None else cu.to(torch.int32).contiguous()
    host = None if keep is None else ctypes.c_void_p(keep.data_ptr())
    lib = N.lib()
    N.check(lib.la_set_sequence_split(1 if split else 0, 256))
    try:
        return int(lib.la_gla_fwd_workspace_size(ctypes.byref(d), N.LA_DTYPE_BF16, host))
    finally:
        N.check(lib.la_set_sequence_split(1, 256))


def _run(x, reverse, g_dev=None):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    if g_dev is not None:
        d["g"] = g_dev
    o, fin, ops = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], d["scale"],
                             d["initial_state"], reverse, x["cu_seqlens"], keep_operands=True)
    torch.cuda.synchronize()
    la.get_device_error()
    return dict(o=o.cpu(), final_state=fin.cpu()), ops


def _ref(x, reverse):
    o, fin = oracle.gla_forward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"], x["scale"],
                                x["initial_state"], reverse, x["cu_seqlens"])
    return dict(o=o, final_state=fin)


@pytest.mark.parametrize("B,T,E", [(1, 3000, 128), (2, 1500, 128), (1, 2500, 64)])
def test_gated_split_forward_matches_oracle(B, T, E):
    x = _inputs(B, T, 2, E, seed=T + E)
    # the split's workspace (segment tables, states, decays) is the larger one
    assert _fwd_ws_bytes(x, True) > _fwd_ws_bytes(x, False) > 0
    for reverse in (False, True):
        got, ops = _run(x, reverse)
        assert ops is None   # per-segment operands are not offered to the backward
        compare(got, _ref(x, reverse), TOL[torch.bfloat16],
                label="gated split B=%d T=%d E=%d rev=%d" % (B, T, E, reverse))


def test_gated_split_packed_with_out_of_range_segments():
    # packed sequences (one shorter than a segment, one empty); head 1's
    # gates leave the chunked form's range over part of the first sequence,
    # so those segments run token by token in both passes
    x = _inputs(1, 0, 2, 128, seqlens=[2100, 0, 700, 100, 37], seed=5)
    x["g"][0, 300:900, 1] = -3.0
    assert _fwd_ws_bytes(x, True) > _fwd_ws_bytes(x, False)
    for reverse in (False, True):
        got, _ = _run(x, reverse)
        compare(got, _ref(x, reverse), TOL[torch.bfloat16], cu=x["cu_seqlens"],
                label="gated split packed rev=%d" % reverse)


def test_gated_split_and_unsplit_agree():
    x = _inputs(1, 3000, 2, 128, seed=9)
    got, _ = _run(x, False)
    N.check(N.lib().la_set_sequence_split(0, 0))
    whole, ops = _run(x, False)
    assert ops is not None   # unsplit: the operands are kept
    for name in got:
        ref = whole[name].float()
        assert (got[name].float() - ref).abs().max() <= 2e-2 * ref.abs().max(), name


def test_gate_without_a_one_row_view_runs_unsplit():
    # a gate whose batch stride is not T times its token stride: the split
    # cannot view the tokens as one row, so the call runs unsplit (correctly)
    x = _inputs(2, 1500, 2, 128, seed=11)
    wide = torch.zeros((2, 1600, 2, 128), device="cuda")
    wide[:, :1500] = x["g"].cuda()
    g_dev = wide[:, :1500]
    assert g_dev.stride(0) != 1500 * g_dev.stride(1)
    for reverse in (False, True):
        got, ops = _run(x, reverse, g_dev)
        assert ops is not None
        compare(got, _ref(x, reverse), TOL[torch.bfloat16],
                label="gated unsplit gate layout rev=%d" % reverse)


def test_gated_split_training_step():
    # recurrent(g=...) with the split forward; the backward recomputes the
    # rescaled operands for the whole sequences
    x = _inputs(1, 2000, 2, 128, seed=13)
    q, k, v, g = (x[n].cuda().requires_grad_() for n in ("q", "k", "v", "g"))
    o, fin = la.recurrent(q, k, v, g=g, g_gamma=x["g_gamma"], softmax_scale=x["scale"])
    ((o.float() * x["do"].cuda().float()).sum()).backward()
    torch.cuda.synchronize()
    ro, rf = oracle.gla_forward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"], x["scale"])
    rq, rk, rv, rg, _ = oracle.gla_backward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"],
                                            x["scale"], x["do"])
    compare(dict(o=o.detach().cpu(), final_state=fin.detach().cpu(), dq=q.grad.cpu(),
                 dk=k.grad.cpu(), dv=v.grad.cpu(), dg=g.grad.cpu()),
            dict(o=ro, final_state=rf, dq=rq, dk=rk, dv=rv, dg=rg), TOL[torch.bfloat16],
            label="gated split training step")


def _bwd_ws_bytes(x, split):
    d = N.LaDims()
    B, T, H, D = x["q"].shape
    E = x["v"].shape[3]
    cu = x["cu_seqlens"]
    d.batch, d.seq_len, d.heads, d.dim_qk, d.dim_v = B, T, H, D, E
    d.num_seqs = 0 if cu is None else len(cu) - 1
    for i in range(3):
        d.qk_strides[i] = x["q"].stride(i)
        d.v_strides[i] = x["v"].stride(i)
    keep = None if cu is None else cu.to(torch.int32).contiguous()
    host = None if keep is None else ctypes.c_void_p(keep.data_ptr())
    lib = N.lib()
    N.check(lib.la_set_sequence_split(1 if split else 0, 256))
    try:
        return int(lib.la_gla_workspace_size(ctypes.byref(d), N.LA_DTYPE_BF16, host, 0))
    finally:
        N.check(lib.la_set_sequence_split(1, 256))


def _full(x, reverse):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, fin = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], d["scale"],
                        d["initial_state"], reverse, x["cu_seqlens"])
    dq, dk, dv, dg, dinit = la.gla_bwd(d["q"], d["k"], d["v"], d["do"], d["g"], d["g_gamma"],
                                       d["scale"], d["initial_state"], d["d_final_state"],
                                       reverse, x["cu_seqlens"])
    torch.cuda.synchronize()
    la.get_device_error()
    out = dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, dg=dg, d_initial_state=dinit)
    return {k: v.cpu() for k, v in out.items()}


def _full_ref(x, reverse):
    ref = _ref(x, reverse)
    dq, dk, dv, dg, dinit = oracle.gla_backward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"],
                                                x["scale"], x["do"], x["initial_state"],
                                                x["d_final_state"], reverse, x["cu_seqlens"])
    ref.update(dq=dq, dk=dk, dv=dv, dg=dg, d_initial_state=dinit)
    return ref


# The backward split: dq~ in two passes around a scan with column decays,
# dv around a scan against the processing order (which gives d_initial_state),
# dk~ from the scanned G transposed, and dg per segment plus each segment's
# offset (the later segments' terms and the final state's term).
@pytest.mark.parametrize("B,T,E", [(1, 3000, 128), (2, 1500, 128), (1, 2500, 64)])
def test_gated_split_backward_matches_oracle(B, T, E):
    x = _inputs(B, T, 2, E, seed=2 * T + E)
    assert _bwd_ws_bytes(x, True) > _bwd_ws_bytes(x, False) > 0
    for reverse in (False, True):
        compare(_full(x, reverse), _full_ref(x, reverse), TOL[torch.bfloat16],
                label="gated split fwd+bwd B=%d T=%d E=%d rev=%d" % (B, T, E, reverse))


def test_gated_split_backward_packed_with_out_of_range_segments():
    # flagged segments (head 1, tokens 300-900 of the first sequence) take
    # their dg from the block scan and their totals from its block sums
    x = _inputs(1, 0, 2, 128, seqlens=[2100, 0, 700, 100, 37], seed=6)
    x["g"][0, 300:900, 1] = -3.0
    assert _bwd_ws_bytes(x, True) > _bwd_ws_bytes(x, False)
    for reverse in (False, True):
        compare(_full(x, reverse), _full_ref(x, reverse), TOL[torch.bfloat16],
                cu=x["cu_seqlens"], label="gated split packed fwd+bwd rev=%d" % reverse)


def test_gated_split_backward_grouped_heads():
    x = _inputs(1, 3000, 4, 128, seed=7)
    G = 2
    kv = dict(x, k=x["k"][:, :, ::G].contiguous(), v=x["v"][:, :, ::G].contiguous())
    rep = dict(x, k=kv["k"].repeat_interleave(G, dim=2), v=kv["v"].repeat_interleave(G, dim=2))
    for reverse in (False, True):
        ref = _full_ref(rep, reverse)
        for name in ("dk", "dv"):
            t = torch.as_tensor(ref[name])
            ref[name] = t.reshape(t.shape[0], t.shape[1], -1, G, t.shape[3]).sum(3)
        compare(_full(kv, reverse), ref, TOL[torch.bfloat16],
                label="gated split grouped rev=%d" % reverse)


def test_gated_split_backward_equals_unsplit_closely():
    x = _inputs(1, 3000, 2, 128, seed=8)
    got = _full(x, False)
    N.check(N.lib().la_set_sequence_split(0, 0))
    whole = _full(x, False)
    for name in got:
        ref = whole[name].float()
        assert (got[name].float() - ref).abs().max() <= 2e-2 * ref.abs().max(), name


def test_gated_split_grouped_packed_out_of_range_both_directions():
    # everything at once: packed sequences (one empty), two query heads per
    # key/value head, one query head's gates out of range over part of the
    # longest sequence, both directions, forward and backward
    x = _inputs(1, 0, 4, 128, seqlens=[2600, 0, 900, 33], seed=15)
    x["g"][0, 1000:1600, 3] = -3.0
    G = 2
    kv = dict(x, k=x["k"][:, :, ::G].contiguous(), v=x["v"][:, :, ::G].contiguous())
    rep = dict(x, k=kv["k"].repeat_interleave(G, dim=2), v=kv["v"].repeat_interleave(G, dim=2))
    for reverse in (False, True):
        ref = _full_ref(rep, reverse)
        for name in ("dk", "dv"):
            t = torch.as_tensor(ref[name])
            ref[name] = t.reshape(t.shape[0], t.shape[1], -1, G, t.shape[3]).sum(3)
        compare(_full(kv, reverse), ref, TOL[torch.bfloat16], cu=x["cu_seqlens"],
                label="gated split grouped packed rev=%d" % reverse)


def test_gated_split_packed_value_width_64():
    x = _inputs(1, 0, 2, 64, seqlens=[1800, 300, 0, 2500], seed=16)
    for reverse in (False, True):
        compare(_full(x, reverse), _full_ref(x, reverse), TOL[torch.bfloat16],
                cu=x["cu_seqlens"], label="gated split packed E=64 rev=%d" % reverse)
