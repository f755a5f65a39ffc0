"""Grouped key/value heads: H query heads sharing H_kv key/value heads.

The reference result is the oracle run with every key/value head repeated
for its G = H / H_kv query heads (the definition of sharing), with the
gradient of a shared head the sum of its copies' gradients (the chain rule
through the repetition).  Checked for the chunked tensor-core path (bf16,
D = 128, groups of 2, 3, 4 and 8), the CUDA-core path (fp32), the
token-by-token path (short sequences), packed sequences, both directions,
and with the sequence split.
"""
import math

import pytest
import torch

import linear_attention_head_gb300 as la
import workloads as W
from linear_attention_head_gb300 import _native as N
from parity import TOL, compare, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


def _grouped(B, T, H, Hkv, D, dtype, seqlens=None, seed=0):
    w = W.Workload("gqa", B, T if seqlens is None else sum(seqlens), H, D, D, dtype,
                   W.alibi_g_gamma(H), 1.0 / math.sqrt(D), seqlens=seqlens, init_std=0.2,
                   dfinal_std=0.2)
    x = W.make_inputs(w, seed=seed)
    G = H // Hkv
    kv = dict(x, k=x["k"][:, :, ::G].contiguous(), v=x["v"][:, :, ::G].contiguous())
    rep = dict(x, k=kv["k"].repeat_interleave(G, dim=2), v=kv["v"].repeat_interleave(G, dim=2))
    return kv, rep, G


def _reference(rep, G, reverse):
    ref = oracle_run(rep, reverse)
    for name in ("dk", "dv"):
        t = torch.as_tensor(ref[name])
        B, T, H, X = t.shape
        ref[name] = t.reshape(B, T, H // G, G, X).sum(3)
    return ref


@pytest.mark.parametrize("T,H,Hkv,D,dtype", [
    (300, 4, 2, 128, torch.bfloat16),     # tensor-core chunked kernels, groups of 2
    (300, 8, 2, 128, torch.bfloat16),     # groups of 4
    (300, 8, 1, 128, torch.bfloat16),     # one key/value head for all queries
    (300, 6, 2, 128, torch.bfloat16),     # groups of 3
    (200, 4, 2, 64, torch.float32),       # CUDA-core chunked kernels
    (7, 6, 3, 128, torch.bfloat16),       # token-by-token kernels
])
def test_grouped_heads_match_oracle(T, H, Hkv, D, dtype):
    kv, rep, G = _grouped(2, T, H, Hkv, D, dtype, seed=T + H)
    for reverse in (False, True):
        compare(gpu_run(kv, reverse), _reference(rep, G, reverse), TOL[dtype],
                label="T=%d H=%d Hkv=%d rev=%d" % (T, H, Hkv, reverse))


def test_grouped_heads_streamed_decode():
    # 20 x 16 = 320 (sequence, head) blocks of 9 tokens, 4 query heads per
    # key/value head: the streamed tensor-core decode reads the shared rows
    assert torch.cuda.get_device_properties(0).multi_processor_count <= 160
    kv, rep, G = _grouped(20, 9, 16, 4, 128, torch.bfloat16, seed=19)
    for reverse in (False, True):
        compare(gpu_run(kv, reverse), _reference(rep, G, reverse), TOL[torch.bfloat16],
                label="streamed decode rev=%d" % reverse)


def test_grouped_heads_packed():
    lens = [130, 0, 257, 5]
    kv, rep, G = _grouped(1, 0, 4, 2, 128, torch.bfloat16, seqlens=lens, seed=9)
    for reverse in (False, True):
        compare(gpu_run(kv, reverse), _reference(rep, G, reverse), TOL[torch.bfloat16],
                cu=kv["cu_seqlens"], label="packed rev=%d" % reverse)


def test_grouped_heads_with_sequence_split():
    N.check(N.lib().la_set_sequence_split(1, 256))
    try:
        kv, rep, G = _grouped(1, 3000, 4, 2, 128, torch.bfloat16, seed=11)
        compare(gpu_run(kv), _reference(rep, G, False), TOL[torch.bfloat16], label="split")
    finally:
        N.check(N.lib().la_set_sequence_split(1, 0))


def test_grouped_heads_autograd_and_shape_checks():
    kv, rep, G = _grouped(1, 100, 4, 2, 64, torch.float32, seed=13)
    q, k, v = (kv[n].cuda().requires_grad_() for n in ("q", "k", "v"))
    o, _ = la.recurrent(q, k, v, g_gamma=kv["g_gamma"], softmax_scale=kv["scale"])
    o.backward(kv["do"].cuda())
    ref = _reference(dict(rep, initial_state=None, d_final_state=None), G, False)
    compare(dict(o=o.detach().cpu(), dq=q.grad.cpu(), dk=k.grad.cpu(), dv=v.grad.cpu()),
            {n: ref[n] for n in ("o", "dq", "dk", "dv")}, TOL[torch.float32], label="autograd")
    with pytest.raises(ValueError):
        la.la_fwd(q.detach(), k.detach()[:, :, :1].expand(-1, -1, 3, -1), v.detach()[:, :, :1]
                  .expand(-1, -1, 3, -1), kv["g_gamma"], 1.0)
    with pytest.raises(ValueError):
        la.lightning_attn(q.detach(), k.detach(), v.detach(), 0, 2)
