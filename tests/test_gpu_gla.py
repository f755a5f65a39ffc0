"""Gated form (GLA): a per-key log-decay gate g [B,T,H,D] on top of g_gamma.

Checked against the fp64 oracle's gated recurrence (tests/test_oracle_gla.py
pins it) for the forward (o, final state) and the backward (dq, dk, dv, dg,
d_initial_state), bf16 and fp32, both directions, packed sequences with an
empty one, and through autograd (`recurrent(g=...)`, `recurrent_gla`).
"""
import math

import pytest
import torch

import linear_attention_head_gb300 as la
import oracle
import workloads as W
from linear_attention_head_gb300 import _native as N
from parity import TOL, compare, compare_gated as _compare_gla

pytestmark = pytest.mark.gpu


def _inputs(B, T, H, D, E, dtype, seqlens=None, seed=0, gate_scale=0.3):
    w = W.Workload("gla", B, T if seqlens is None else sum(seqlens), H, D, E, dtype,
                   W.alibi_g_gamma(H), 1.0 / math.sqrt(D), seqlens=seqlens, init_std=0.2,
                   dfinal_std=0.2)
    x = W.make_inputs(w, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1000)
    x["g"] = -gate_scale * torch.rand(x["q"].shape, generator=gen)
    return x


def _gpu(x, reverse, chunked=True):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, fin = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], d["scale"],
                        d["initial_state"], reverse, x["cu_seqlens"], chunked=chunked)
    dq, dk, dv, dg, dinit = la.gla_bwd(d["q"], d["k"], d["v"], d["do"], d["g"], d["g_gamma"],
                                       d["scale"], d["initial_state"], d["d_final_state"],
                                       reverse, x["cu_seqlens"], chunked=chunked)
    torch.cuda.synchronize()
    la.get_device_error()
    out = dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, dg=dg, d_initial_state=dinit)
    return {k: v.cpu() for k, v in out.items()}


def _oracle(x, reverse):
    o, fin = oracle.gla_forward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"], x["scale"],
                                x["initial_state"], reverse, x["cu_seqlens"])
    dq, dk, dv, dg, dinit = oracle.gla_backward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"],
                                                x["scale"], x["do"], x["initial_state"],
                                                x["d_final_state"], reverse, x["cu_seqlens"])
    return dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, dg=dg, d_initial_state=dinit)


@pytest.mark.parametrize("T,D,E,dtype", [(300, 128, 128, torch.bfloat16),
                                         (200, 64, 64, torch.float32),
                                         (37, 48, 80, torch.bfloat16)])
def test_gated_matches_oracle(T, D, E, dtype):
    x = _inputs(2, T, 3, D, E, dtype, seed=T)
    for reverse in (False, True):
        label = "gla T=%d rev=%d" % (T, reverse)
        plain, cond = _compare_gla(_gpu(x, reverse), _oracle(x, reverse), x, reverse, TOL[dtype],
                                   label)
        print("%s: dg plain %.2e, conditioned %.2e" % (label, plain, cond))


# dg's plain error, max|x - ref| / max|ref| per (sequence, head), beside the
# conditioned one, at 2000 tokens, on the tensor cores and token by token.
# dg adds up one term per token; formed from bf16-rounded dq, dk it read
# 0.022 here (0.04-0.05 at 8192 tokens), a random walk of the rounding.  The
# kernels take the gradients in fp32, and the chunked form takes each term
# from its rounded operands and their own gradients, so that only bounded
# errors remain: about 0.004 on the tensor cores (the operands' rounding, as
# for dq and dk themselves), fp32 rounding token by token.
@pytest.mark.parametrize("chunked,bound", [(True, 1e-2), (False, 1e-3)])
def test_gated_dg_plain_error_at_2000_tokens(chunked, bound):
    x = _inputs(2, 2000, 3, 128, 128, torch.bfloat16, seed=2000)
    for reverse in (False, True):
        label = "gla T=2000 chunked=%d rev=%d" % (chunked, reverse)
        plain, cond = _compare_gla(_gpu(x, reverse, chunked), _oracle(x, reverse), x, reverse,
                                   TOL[torch.bfloat16], label)
        print("%s: dg plain %.2e, conditioned %.2e" % (label, plain, cond))
        assert plain <= bound, (label, plain)


def test_gated_packed_sequences():
    lens = [70, 0, 133, 5]
    x = _inputs(1, 0, 2, 64, 64, torch.float32, seqlens=lens, seed=3)
    for reverse in (False, True):
        _compare_gla(_gpu(x, reverse), _oracle(x, reverse), x, reverse, TOL[torch.float32],
                     "gla packed rev=%d" % reverse)


def test_gated_autograd_and_recurrent_gla():
    x = _inputs(1, 120, 2, 64, 64, torch.float32, seed=5)
    q, k, v, g = (x[n].cuda().requires_grad_() for n in ("q", "k", "v", "g"))
    o, fin = la.recurrent_gla(q, k, v, g=g, g_gamma=x["g_gamma"], softmax_scale=x["scale"])
    (o * x["do"].cuda()).sum().backward()
    ref_o, _ = oracle.gla_forward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"], x["scale"])
    rq, rk, rv, rg, _ = oracle.gla_backward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"],
                                            x["scale"], x["do"])
    compare(dict(o=o.detach().cpu(), dq=q.grad.cpu(), dk=k.grad.cpu(), dv=v.grad.cpu(),
                 dg=g.grad.cpu()),
            dict(o=ref_o, dq=rq, dk=rk, dv=rv, dg=rg), TOL[torch.float32], label="autograd")


def test_gate_of_zero_equals_the_ungated_path():
    x = _inputs(2, 260, 2, 128, 128, torch.bfloat16, seed=7)
    x["g"] = torch.zeros_like(x["g"])
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o1, f1 = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], d["scale"],
                        d["initial_state"])
    o2, f2 = la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], d["scale"], d["initial_state"])
    # the chunked tensor-core path rounds its MMA operands to bf16, the gated
    # path runs in fp32: both meet the bf16 parity bound against the oracle
    assert (o1.float() - o2.float()).abs().max() <= 2e-2 * o2.float().abs().max()
    assert (f1 - f2).abs().max() <= 2e-2 * f2.abs().max()


@pytest.mark.parametrize("T", [1, 3])
def test_gated_decode_streamed(T):
    # 20 x 16 = 320 (sequence, head) blocks of at most 4 tokens: the gated
    # forward takes the streamed decode kernel (row gate)
    assert torch.cuda.get_device_properties(0).multi_processor_count <= 160
    x = _inputs(20, T, 16, 128, 128, torch.bfloat16, seed=40 + T)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    for reverse in (False, True):
        o, fin = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], d["scale"],
                            d["initial_state"], reverse)
        torch.cuda.synchronize()
        la.get_device_error()
        ro, rf = oracle.gla_forward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"], x["scale"],
                                    x["initial_state"], reverse)
        compare(dict(o=o.cpu(), final_state=fin.cpu()), dict(o=ro, final_state=rf),
                TOL[torch.bfloat16], label="gated streamed T=%d rev=%d" % (T, reverse))


def _fwd_only(x, reverse, chunked=True):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, fin = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], d["scale"],
                        d["initial_state"], reverse, x["cu_seqlens"], chunked=chunked)
    torch.cuda.synchronize()
    la.get_device_error()
    ro, rf = oracle.gla_forward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"], x["scale"],
                                x["initial_state"], reverse, x["cu_seqlens"])
    return dict(o=o.cpu(), final_state=fin.cpu()), dict(o=ro, final_state=rf)


# The chunked tensor-core form (bf16, D = 128, E in {64, 128}, > 16 tokens):
# several chunks and a ragged tail, both directions, with and without an
# initial state.  At E = 64 the backward's dq~ and dk~ sweeps hold the 64
# value channels on TMEM lanes (the state's rows) and the 128 gated key
# channels as columns.
@pytest.mark.parametrize("T,E", [(300, 128), (1000, 128), (517, 64), (300, 64)])
@pytest.mark.parametrize("init", [0.2, 0.0])
def test_gated_chunked_matches_oracle(T, E, init):
    x = _inputs(2, T, 3, 128, E, torch.bfloat16, seed=T + E)
    if init == 0.0:
        x["initial_state"] = None
    for reverse in (False, True):
        label = "chunked T=%d E=%d rev=%d" % (T, E, reverse)
        _compare_gla(_gpu(x, reverse), _oracle(x, reverse), x, reverse, TOL[torch.bfloat16],
                     label)


def test_gated_backward_at_e64_runs_the_chunked_form():
    # the chunked backward launches the pre-pass, three tensor-core sweeps and
    # the rescaling pass on top of the token-by-token launches (which find
    # every pair done and return): at least five more launches than the
    # token-by-token backward, and different rounding
    lib = N.lib()
    x = _inputs(1, 400, 2, 128, 64, torch.bfloat16, seed=64)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    got, counts = {}, {}
    for chunked in (True, False):
        n0 = lib.la_launch_count()
        got[chunked] = la.gla_bwd(d["q"], d["k"], d["v"], d["do"], d["g"], d["g_gamma"],
                                  d["scale"], d["initial_state"], d["d_final_state"],
                                  chunked=chunked)
        torch.cuda.synchronize()
        counts[chunked] = lib.la_launch_count() - n0
    assert counts[True] >= counts[False] + 5, counts
    assert not torch.equal(got[True][0], got[False][0])


def test_gated_chunked_packed_sequences():
    lens = [70, 0, 300, 129, 5, 256, 17]
    x = _inputs(1, 0, 2, 128, 128, torch.bfloat16, seqlens=lens, seed=8)
    for reverse in (False, True):
        _compare_gla(_gpu(x, reverse), _oracle(x, reverse), x, reverse, TOL[torch.bfloat16],
                     "chunked packed rev=%d" % reverse)


def test_gated_chunked_strong_gates_run_token_by_token():
    # head 1's gates (-3 per token) put the running sums out of the chunked
    # form's range: that (sequence, head) runs token by token in the same
    # call, the others on the tensor cores; both agree with the oracle, and
    # with the all-token-by-token call
    x = _inputs(2, 400, 3, 128, 128, torch.bfloat16, seed=9)
    x["g"][:, :, 1] = -3.0
    x["g"][1, 100:160, 2] = -4.0   # one chunk of one sequence out of range
    for reverse in (False, True):
        _compare_gla(_gpu(x, reverse), _oracle(x, reverse), x, reverse, TOL[torch.bfloat16],
                     "mixed rev=%d" % reverse)
        got, ref = _fwd_only(x, reverse)
        tok, _ = _fwd_only(x, reverse, chunked=False)
        compare(tok, ref, TOL[torch.bfloat16], label="token rev=%d" % reverse)


def test_gated_backward_reuses_forward_operands():
    # gla_fwd(keep_operands=True) hands its rescaled q, k to gla_bwd, which
    # skips computing them; out-of-range pairs (head 1) keep their flags
    x = _inputs(2, 400, 3, 128, 128, torch.bfloat16, seed=12)
    x["g"][:, :, 1] = -3.0
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    for reverse in (False, True):
        o, fin, ops = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], d["scale"],
                                 d["initial_state"], reverse, keep_operands=True)
        assert ops is not None
        dq, dk, dv, dg, dinit = la.gla_bwd(d["q"], d["k"], d["v"], d["do"], d["g"],
                                           d["g_gamma"], d["scale"], d["initial_state"],
                                           d["d_final_state"], reverse, operands=ops)
        torch.cuda.synchronize()
        la.get_device_error()
        got = dict(o=o, final_state=fin, dq=dq, dk=dk, dv=dv, dg=dg, d_initial_state=dinit)
        _compare_gla({k: v.cpu() for k, v in got.items()}, _oracle(x, reverse), x, reverse,
                     TOL[torch.bfloat16], "reused operands rev=%d" % reverse)
    # the token-by-token forward leaves no operands to reuse
    _, _, none = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], d["scale"],
                            keep_operands=True, chunked=False)
    assert none is None


def test_gated_autograd_chunked_bf16():
    # recurrent_gla's autograd path at the chunked form's sizes (the backward
    # reuses the forward's operands)
    x = _inputs(1, 300, 2, 128, 128, torch.bfloat16, seed=13)
    q, k, v, g = (x[n].cuda().requires_grad_() for n in ("q", "k", "v", "g"))
    o, fin = la.recurrent_gla(q, k, v, g=g, g_gamma=x["g_gamma"], softmax_scale=x["scale"])
    ((o.float() * x["do"].cuda().float()).sum()).backward()
    torch.cuda.synchronize()
    ref_o, ref_f = oracle.gla_forward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"], x["scale"])
    rq, rk, rv, rg, _ = oracle.gla_backward(x["q"], x["k"], x["v"], x["g"], x["g_gamma"],
                                            x["scale"], x["do"])
    y = dict(x, initial_state=None, d_final_state=None)
    _compare_gla(dict(o=o.detach().cpu(), dq=q.grad.cpu(), dk=k.grad.cpu(), dv=v.grad.cpu(),
                      dg=g.grad.cpu()),
                 dict(o=ref_o, final_state=ref_f, dq=rq, dk=rk, dv=rv, dg=rg), y, False,
                 TOL[torch.bfloat16], "autograd chunked")


def test_gated_chunked_strong_decay_in_range():
    # running sums near the chunked form's range (about -127 per 128-token
    # chunk: g_gamma -0.84 plus the gate) without leaving it: the state's two
    # factors at a chunk boundary, exp(B - r) and the next exp(r), multiply to
    # below fp32's range and must be applied one after the other
    x = _inputs(2, 700, 2, 128, 128, torch.bfloat16, seed=21)
    x["g_gamma"] = torch.tensor([-2.0 ** -0.25, -0.5], dtype=torch.float32)
    for reverse in (False, True):
        _compare_gla(_gpu(x, reverse), _oracle(x, reverse), x, reverse, TOL[torch.bfloat16],
                     "strong in range rev=%d" % reverse)


def _grouped_gated(B, T, H, Hkv, D, E, dtype, seqlens=None, seed=0):
    """Gated inputs with H_kv key/value heads (each repeated for its G query
    heads in the oracle's copy); the gate is the query heads'."""
    x = _inputs(B, T, H, D, E, dtype, seqlens=seqlens, seed=seed)
    G = H // Hkv
    kv = dict(x, k=x["k"][:, :, ::G].contiguous(), v=x["v"][:, :, ::G].contiguous())
    rep = dict(x, k=kv["k"].repeat_interleave(G, dim=2), v=kv["v"].repeat_interleave(G, dim=2))
    return kv, rep, G


def _group_sums(ref, G):
    for name in ("dk", "dv"):
        t = torch.as_tensor(ref[name])
        B, T, H, X = t.shape
        ref[name] = t.reshape(B, T, H // G, G, X).sum(3)
    return ref


# Grouped key/value heads with the gate (ejkernel `recurrent`: key and value
# with num_kv_heads heads, g with the queries' heads): the oracle on the
# repeated heads, dk and dv summed over each group.
@pytest.mark.parametrize("T,H,Hkv,D,E,dtype,chunked", [
    (300, 6, 2, 128, 128, torch.bfloat16, True),    # chunked form, groups of 3
    (300, 4, 1, 128, 128, torch.bfloat16, False),   # token by token, one key/value head
    (517, 4, 2, 128, 64, torch.bfloat16, True),     # chunked forward, E = 64
    (200, 4, 2, 64, 64, torch.float32, True),       # fp32 tokens
    (9, 8, 2, 128, 128, torch.bfloat16, True),      # short sequences
])
def test_gated_grouped_heads_match_oracle(T, H, Hkv, D, E, dtype, chunked):
    kv, rep, G = _grouped_gated(2, T, H, Hkv, D, E, dtype, seed=T + H)
    for reverse in (False, True):
        ref = _group_sums(_oracle(rep, reverse), G)
        compare(_gpu(kv, reverse, chunked), ref, TOL[dtype],
                label="gated grouped T=%d H=%d Hkv=%d E=%d chunked=%d rev=%d"
                % (T, H, Hkv, E, chunked, reverse))


def test_gated_grouped_heads_packed_with_strong_gates():
    # packed sequences (one empty) and query head 1 gated by -3 per token: its
    # long sequences leave the chunked form's range and run token by token
    # beside the tensor-core pairs, and both parts meet in the group sums.
    # Sharing a key/value head changes no query head's arithmetic: o, the
    # states, dq and dg equal those of the same call on repeated heads bit
    # for bit, and dk, dv are the oracle's group sums.
    kv, rep, G = _grouped_gated(1, 0, 4, 2, 128, 128, torch.bfloat16,
                                seqlens=[70, 0, 300, 129, 5], seed=17)
    for x in (kv, rep):
        x["g"] = x["g"].clone()
        x["g"][:, :, 1] = -3.0
    for reverse in (False, True):
        got, same = _gpu(kv, reverse), _gpu(rep, reverse)
        for name in ("o", "final_state", "dq", "dg", "d_initial_state"):
            assert torch.equal(got[name], same[name]), name
        ref = _oracle(rep, reverse)
        # the 5-token sequence (index 4) stays in range on head 1, on the
        # tensor cores: its dg (max 0.37) is a near-cancelling sum of terms
        # up to about 3, each with the bf16 operands' error of dq~ and dk~, so
        # the plain ratio reads about 0.04 there; held to the conditioned bound
        plain, cond = _compare_gla(same, ref, rep, reverse, TOL[torch.bfloat16],
                                   "gated repeated packed rev=%d" % reverse,
                                   plain_dg_except={(4, 1)})
        print("rev=%d: dg plain %.2e elsewhere, conditioned %.2e" % (reverse, plain, cond))
        ref = _group_sums(ref, G)
        compare(dict(dk=got["dk"], dv=got["dv"]), dict(dk=ref["dk"], dv=ref["dv"]),
                TOL[torch.bfloat16], cu=kv["cu_seqlens"], label="gated grouped packed rev=%d"
                % reverse)


def test_gated_grouped_heads_autograd():
    # recurrent(g=...) with grouped keys and values: the forward keeps its
    # operands for the backward; key.grad and value.grad have the shared
    # heads' shape
    kv, rep, G = _grouped_gated(1, 300, 4, 2, 128, 128, torch.bfloat16, seed=23)
    q, k, v, g = (kv[n].cuda().requires_grad_() for n in ("q", "k", "v", "g"))
    o, fin = la.recurrent(q, k, v, g=g, g_gamma=kv["g_gamma"], softmax_scale=kv["scale"])
    ((o.float() * kv["do"].cuda().float()).sum()).backward()
    torch.cuda.synchronize()
    assert k.grad.shape == k.shape and v.grad.shape == v.shape
    ro, _ = oracle.gla_forward(rep["q"], rep["k"], rep["v"], rep["g"], rep["g_gamma"],
                               rep["scale"])
    rq, rk, rv, rg, _ = oracle.gla_backward(rep["q"], rep["k"], rep["v"], rep["g"],
                                            rep["g_gamma"], rep["scale"], rep["do"])
    ref = _group_sums(dict(o=ro, dq=rq, dk=rk, dv=rv, dg=rg), G)
    compare(dict(o=o.detach().cpu(), dq=q.grad.cpu(), dk=k.grad.cpu(), dv=v.grad.cpu(),
                 dg=g.grad.cpu()), ref, TOL[torch.bfloat16], label="gated grouped autograd")


def test_gated_keys_with_strides_of_their_own_through_the_c_abi():
    # kv_heads = H with k (and dk) head-major while q is token-major: the
    # pre-pass reads k, and the rescaling pass writes dk, at k's own strides.
    # Same values as the call on a token-major k, bit for bit.
    import ctypes
    from linear_attention_head_gb300 import api as A
    x = _inputs(2, 300, 3, 128, 128, torch.bfloat16, seed=31)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    ref_o, ref_f = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], d["scale"],
                              d["initial_state"])
    ref_b = la.gla_bwd(d["q"], d["k"], d["v"], d["do"], d["g"], d["g_gamma"], d["scale"],
                       d["initial_state"], d["d_final_state"])
    B, T, H, D = d["q"].shape
    k_hm = d["k"].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)   # [B,T,H,D] view
    dk_hm = torch.empty((B, H, T, D), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)
    dims = N.LaDims()
    dims.batch, dims.seq_len, dims.heads, dims.dim_qk, dims.dim_v = B, T, H, D, 128
    dims.num_seqs, dims.kv_heads = 0, H
    for i in range(3):
        dims.qk_strides[i] = d["q"].stride(i)
        dims.v_strides[i] = d["v"].stride(i)
        dims.k_strides[i] = k_hm.stride(i)
        dims.kv_v_strides[i] = d["v"].stride(i)
    lib, st = N.lib(), A._stream(torch.device("cuda"))
    o, fin = torch.empty_like(d["v"]), torch.empty_like(ref_f)
    nb = int(lib.la_gla_fwd_workspace_size(ctypes.byref(dims), N.LA_DTYPE_BF16, None))
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    written = ctypes.c_int32(0)
    N.check(lib.la_gla_fwd(ctypes.byref(dims), N.LA_DTYPE_BF16, A._ptr(d["q"]), A._ptr(k_hm),
                           A._ptr(d["v"]), A._ptr(d["g"]), A._strides3(d["g"]),
                           A._ptr(d["g_gamma"]), float(d["scale"]), A._ptr(d["initial_state"]),
                           0, None, None, A._ptr(o), A._ptr(fin), A._ptr(ws), nb,
                           ctypes.byref(written), st))
    assert written.value == 1
    dq, dv = torch.empty_like(d["q"]), torch.empty_like(d["v"])
    dg, dinit = torch.empty_like(d["g"]), torch.empty_like(ref_f)
    nb2 = int(lib.la_gla_workspace_size(ctypes.byref(dims), N.LA_DTYPE_BF16, None, 0))
    ws2 = torch.empty(nb2, dtype=torch.uint8, device="cuda")
    N.check(lib.la_gla_bwd(ctypes.byref(dims), N.LA_DTYPE_BF16, A._ptr(d["q"]), A._ptr(k_hm),
                           A._ptr(d["v"]), A._ptr(d["do"]), A._ptr(d["g"]), A._strides3(d["g"]),
                           A._ptr(d["g_gamma"]), float(d["scale"]), A._ptr(d["initial_state"]),
                           A._ptr(d["d_final_state"]), 0, None, None, A._ptr(dq), A._ptr(dk_hm),
                           A._ptr(dv), A._ptr(dg), A._ptr(dinit), A._ptr(ws2), nb2, None, 0, st))
    torch.cuda.synchronize()
    la.get_device_error()
    got = dict(o=o, final_state=fin, dq=dq, dk=dk_hm, dv=dv, dg=dg, d_initial_state=dinit)
    ref = dict(o=ref_o, final_state=ref_f, dq=ref_b[0], dk=ref_b[1], dv=ref_b[2], dg=ref_b[3],
               d_initial_state=ref_b[4])
    for name in got:
        assert torch.equal(got[name], ref[name]), name
