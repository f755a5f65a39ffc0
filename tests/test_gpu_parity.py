"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on
the same seeded inputs, element by element, at the tolerances of the workload
definitions: max relative error <= 2e-2 for bf16 token tensors and <= 1e-4 for
fp32 (per (sequence, head) slice, tests/parity.py), final and initial-state
gradients included.  Full-size workloads compare a sample of heads that the
oracle computes on its own; everything else compares every element.
"""
import math

import numpy as np
import pytest
import torch

import linear_attention_head_gb300 as la
import workloads as W
from parity import TOL, compare, gpu_run, oracle_run, take_heads, take_out

pytestmark = pytest.mark.gpu


def test_tiny_fp32_forward():
    w = W.tiny_fp32()
    x = W.make_inputs(w, seed=0)
    got = gpu_run(x, backward=False)
    compare(got, oracle_run(x, backward=False), TOL[torch.float32], label=w.name)


@pytest.mark.parametrize("reverse", [False, True])
def test_small_bf16_fwd_bwd(reverse):
    w = W.small_bf16()
    x = W.make_inputs(w, seed=0)
    got = gpu_run(x, reverse)
    compare(got, oracle_run(x, reverse), TOL[torch.bfloat16], label=w.name)


@pytest.mark.parametrize("n", [512, 1024, 2048, 4096])
def test_sweep_shape_full_compare(n):
    w = W.sweep_bf16(n)
    x = W.make_inputs(w, seed=0)
    got = gpu_run(x)
    heads = [0, 13, 31]
    compare(take_out(got, heads), oracle_run(take_heads(x, heads)), TOL[torch.bfloat16],
            label=w.name)


@pytest.mark.parametrize("n", [8192, 16384, 32768])
def test_sweep_shape_sampled(n):
    w = W.sweep_bf16(n)
    x = W.make_inputs(w, seed=0)
    got = gpu_run(x)
    heads, rows = [0, 31], [0, 3]
    compare(take_out(got, heads, rows), oracle_run(take_heads(x, heads, rows)),
            TOL[torch.bfloat16], label=w.name)


def test_d192_fwd_bwd():
    w = W.d192_bf16()
    x = W.make_inputs(w, seed=0)
    got = gpu_run(x)
    heads = [0, 11]
    compare(take_out(got, heads), oracle_run(take_heads(x, heads)), TOL[torch.bfloat16],
            label=w.name)


@pytest.mark.parametrize("reverse", [False, True])
def test_varlen_with_states(reverse):
    w = W.varlen_bf16(seed=0)
    x = W.make_inputs(w, seed=0)
    got = gpu_run(x, reverse)
    heads = [0, 7, 15]
    compare(take_out(got, heads), oracle_run(take_heads(x, heads), reverse),
            TOL[torch.bfloat16], cu=x["cu_seqlens"], label=w.name)


# ---- edge cases -------------------------------------------------------------

def _custom(B, T, H, D, E, dtype, seqlens=None, init=0.0, dfin=0.0, g=None, scale=None):
    g = W.alibi_g_gamma(H) if g is None else g
    return W.Workload("custom", B, T if seqlens is None else sum(seqlens), H, D, E, dtype, g,
                      scale if scale is not None else 1.0 / math.sqrt(D), seqlens=seqlens,
                      init_std=init, dfinal_std=dfin)


@pytest.mark.parametrize("T", [1, 5, 31, 32, 33, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.float32, 64),
                                     (torch.bfloat16, 128)])
def test_ragged_lengths(T, dtype, D):
    w = _custom(2, T, 3, D, D, dtype, init=0.3, dfin=0.3,
                g=torch.tensor([0.0, -0.05, -1.0]))
    x = W.make_inputs(w, seed=T)
    for reverse in (False, True):
        compare(gpu_run(x, reverse), oracle_run(x, reverse), TOL[dtype],
                label="T=%d rev=%d" % (T, reverse))


@pytest.mark.parametrize("D,E", [(32, 32), (64, 128), (128, 64), (128, 128), (192, 192),
                                 (256, 256), (16, 48), (80, 96), (1, 1), (64, 64), (192, 128),
                                 (128, 192), (256, 64)])
def test_head_dims(D, E):
    w = _custom(1, 200, 2, D, E, torch.bfloat16, init=0.2, dfin=0.2)
    x = W.make_inputs(w, seed=D * 1000 + E)
    compare(gpu_run(x), oracle_run(x), TOL[torch.bfloat16], label="D=%d E=%d" % (D, E))


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.float32, 64),
                                     (torch.bfloat16, 128)])
def test_packed_with_empty_and_short_sequences(dtype, D):
    lens = [0, 1, 130, 0, 64, 257, 3, 128, 129]
    if True:
        w = _custom(1, 0, 4, D, D, dtype, seqlens=lens, init=0.1, dfin=0.1)
        x = W.make_inputs(w, seed=5)
        for reverse in (False, True):
            got = gpu_run(x, reverse)
            ref = oracle_run(x, reverse)
            compare(got, ref, TOL[dtype], cu=x["cu_seqlens"], label="packed rev=%d" % reverse)
            # zero-length sequences pass their states through unchanged
            for n in (0, 3):
                assert torch.equal(got["final_state"][n], x["initial_state"][n])
                assert torch.equal(got["d_initial_state"][n], x["d_final_state"][n])


def test_head_major_layout_and_lightning2_call():
    # OpenNLPLab README: q, k, v as (b, h, n, d), slopes s, o = lightning_attn_func(q, k, v, s)
    b, h, n, d, e = 2, 4, 300, 64, 64
    gen = torch.Generator().manual_seed(3)
    qk_shape, v_shape = (b, h, n, d), (b, h, n, e)
    q, k, v = (torch.randn(shape, generator=gen).bfloat16()
               for shape in (qk_shape, qk_shape, v_shape))
    s = -W.alibi_g_gamma(h)
    o = la.lightning_attn_func(q.cuda(), k.cuda(), v.cuda(), s.cuda())
    ref, _ = oracle_run(dict(q=q.transpose(1, 2), k=k.transpose(1, 2), v=v.transpose(1, 2),
                             g_gamma=-s, scale=1.0, initial_state=None, cu_seqlens=None),
                        backward=False).values()
    compare(dict(o=o.transpose(1, 2).cpu()), dict(o=ref), TOL[torch.bfloat16],
            label="head-major")


def test_autograd_matches_la_bwd():
    w = _custom(1, 150, 2, 64, 64, torch.bfloat16, init=0.1, dfin=0.0)
    x = W.make_inputs(w, seed=9)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    q, k, v = (d[n].clone().requires_grad_() for n in ("q", "k", "v"))
    init = d["initial_state"].clone().requires_grad_()
    o, fin = la.recurrent(q, k, v, g_gamma=d["g_gamma"], softmax_scale=w.scale,
                          initial_state=init)
    (o.float() * d["do"].float()).sum().backward()
    ref = oracle_run(dict(x, d_final_state=None))
    got = dict(o=o.detach().cpu(), final_state=fin.detach().cpu(), dq=q.grad.cpu(),
               dk=k.grad.cpu(), dv=v.grad.cpu(), d_initial_state=init.grad.cpu())
    compare(got, ref, TOL[torch.bfloat16], label="autograd")


def test_lightning_attn_docstring_example_closed_form():
    # ejkernel lightning_attn example: ones (2, 2048, 8, 64), layer 5 of 12
    ones = torch.ones((2, 2048, 8, 64), dtype=torch.bfloat16, device="cuda")
    o, fin = la.lightning_attn(ones, ones, ones, layer_idx=5, num_layers=12)
    g = la.lightning_g_gamma(8, 5, 12).double().numpy()
    t = np.arange(2048)
    for h in range(8):
        gam = math.exp(g[h])
        ref = (64 ** -0.5) * 64 * ((t + 1) if gam == 1 else (1 - gam ** (t + 1)) / (1 - gam))
        got = o[0, :, h, 0].float().cpu().double().numpy()
        assert np.max(np.abs(got - ref)) / np.max(ref) < 2e-2


def test_empty_batch_and_zero_length():
    q = torch.zeros((0, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    o, fin = la.la_fwd(q, q, q, torch.zeros(2))
    assert o.shape == q.shape and fin.shape == (0, 2, 64, 64)
    q = torch.zeros((3, 0, 2, 64), dtype=torch.bfloat16, device="cuda")
    init = torch.randn((3, 2, 64, 64), device="cuda")
    o, fin = la.la_fwd(q, q, q, torch.full((2,), -0.5), initial_state=init)
    assert torch.equal(fin, init)


def test_tensor_core_path_is_selected_for_the_benchmark_shape():
    # bf16, d = e = 128, dense token-major: the tcgen05 kernels, not the CUDA-core ones
    assert la.kernel_family(4, 32768, 32, 128, 128) == 1
    assert la.kernel_family(1, 4096, 16, 128, 64) == 1
    assert la.kernel_family(1, 256, 2, 32, 32, dtype=torch.float32) == 0


def test_tensor_core_path_is_selected_for_the_other_head_dims():
    # the small bf16 shape (d = e = 64) and the non-power-of-two one (d = e = 192,
    # the OpenNLPLab README's usage example) run on the tensor cores too
    assert la.kernel_family(2, 2048, 8, 64, 64) == 1
    assert la.kernel_family(2, 2048, 12, 192, 192) == 1
    assert la.kernel_family(1, 300, 2, 256, 64) == 1
    assert la.kernel_family(1, 300, 2, 64, 256) == 1
    # widths that are not multiples of 64 stay on the CUDA-core kernels
    assert la.kernel_family(1, 300, 2, 96, 96) == 0
    assert la.kernel_family(1, 300, 2, 128, 80) == 0


@pytest.mark.parametrize("D,E", [(64, 64), (64, 192), (192, 64), (192, 192), (256, 128),
                                 (128, 256)])
def test_tensor_core_head_dims_packed_states_both_directions(D, E):
    # packed sequences with an empty one and ragged tails, initial state and
    # final-state gradient, forward and reverse: every value tile of every
    # (sequence, head) and every 128-row piece of the state
    lens = [0, 300, 1, 129, 517, 64]
    w = _custom(1, 0, 2, D, E, torch.bfloat16, seqlens=lens, init=0.1, dfin=0.1,
                g=torch.tensor([-0.01, -0.4]))
    x = W.make_inputs(w, seed=D + 7 * E)
    for reverse in (False, True):
        got = gpu_run(x, reverse)
        compare(got, oracle_run(x, reverse), TOL[torch.bfloat16], cu=x["cu_seqlens"],
                label="D=%d E=%d rev=%d" % (D, E, reverse))
        assert torch.equal(got["final_state"][0], x["initial_state"][0])
        assert torch.equal(got["d_initial_state"][0], x["d_final_state"][0])


def test_unaligned_layout_falls_back_and_matches():
    # a channel-contiguous layout whose token stride is not a multiple of 16 bytes
    # cannot be described by TMA; the CUDA-core kernel takes it and must agree.
    w = _custom(2, 200, 3, 128, 128, torch.bfloat16, init=0.2, dfin=0.2)
    x = W.make_inputs(w, seed=21)
    big = {}
    for n in ("q", "k", "v", "do"):
        t = x[n]
        pad = torch.zeros(t.shape[:2] + (t.shape[2] * t.shape[3] + 4,), dtype=t.dtype)
        pad[..., : t.shape[2] * t.shape[3]] = t.reshape(t.shape[0], t.shape[1], -1)
        big[n] = pad.cuda()[..., : t.shape[2] * t.shape[3]].reshape(t.shape)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, fin = la.la_fwd(big["q"], big["k"], big["v"], d["g_gamma"], w.scale, d["initial_state"])
    dq, dk, dv, dinit = la.la_bwd(big["q"], big["k"], big["v"], big["do"], d["g_gamma"], w.scale,
                                  d["initial_state"], d["d_final_state"])
    got = dict(o=o.cpu(), final_state=fin.cpu(), dq=dq.cpu(), dk=dk.cpu(), dv=dv.cpu(),
               d_initial_state=dinit.cpu())
    compare(got, oracle_run(x), TOL[torch.bfloat16], label="unaligned")


def test_repeated_calls_are_deterministic_and_report_no_timeout():
    w = W.sweep_bf16(1024)
    x = W.make_inputs(w, seed=4)
    a = gpu_run(x)
    b = gpu_run(x)
    for n in a:
        assert torch.equal(a[n], b[n]), n
    la.get_device_error()


@pytest.mark.parametrize("D", [64, 128])
def test_longest_first_schedule_is_bit_identical_to_index_order(D):
    # the packed schedule only changes which CTA runs which sequence (the
    # sequence split, which the workspace would also allow, is off here: it
    # sums in another order)
    import ctypes
    from linear_attention_head_gb300 import _native as N
    lens = [5, 300, 0, 129, 64, 1000, 17]
    w = _custom(1, 0, 2, D, D, torch.bfloat16, seqlens=lens, init=0.1)
    x = W.make_inputs(w, seed=31)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    N.check(N.lib().la_set_sequence_split(0, 0))
    try:
        o_sched, f_sched = la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], w.scale,
                                     d["initial_state"], cu_seqlens=x["cu_seqlens"])
    finally:
        N.check(N.lib().la_set_sequence_split(1, 0))
    o_plain = torch.empty_like(o_sched)
    f_plain = torch.empty_like(f_sched)
    dims = N.LaDims()
    B, T, H, Dq = d["q"].shape
    dims.batch, dims.seq_len, dims.heads, dims.dim_qk, dims.dim_v = B, T, H, Dq, D
    dims.num_seqs = len(lens)
    for i in range(3):
        dims.qk_strides[i] = d["q"].stride(i)
        dims.v_strides[i] = d["v"].stride(i)
    cu_dev = x["cu_seqlens"].cuda()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    st = N.lib().la_fwd(ctypes.byref(dims), N.LA_DTYPE_BF16, P(d["q"]), P(d["k"]), P(d["v"]),
                        P(d["g_gamma"]), w.scale, P(d["initial_state"]), 0, P(cu_dev),
                        P(x["cu_seqlens"]), P(o_plain), P(f_plain), None, 0,
                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    N.check(st)
    torch.cuda.synchronize()
    assert torch.equal(o_sched, o_plain)
    assert torch.equal(f_sched, f_plain)
