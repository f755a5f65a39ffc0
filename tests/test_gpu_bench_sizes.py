"""Parity at the sizes bench.py measures its secondary lines at.

Each call runs whole on the GPU, in the configuration the bench times; the
oracle then computes sampled (batch row, head) slices, which must match:
- decode: la_fwd on b64 h32 d=e=128 bf16, one new token, a carried fp32 state
  (the streamed decode kernel);
- the sequence split: la_fwd + la_bwd on b1 h8 n262144 d=e=128 bf16;
- grouped key/value heads: b4 h32, 8 key/value heads, n32768, d=e=128 bf16
  (the oracle runs each sampled query head with its key/value head repeated,
  a shared head's gradients the sum over its group);
- the gated form: gla_fwd + gla_bwd on b4 h32 n8192 d=e=128 bf16 with the
  bench's gate recipe (the chunked tensor-core form).
"""

import pytest
import torch

import linear_attention_head_gb300 as la
import oracle
import workloads as W
from parity import TOL, compare, compare_gated, take_heads, take_out

pytestmark = pytest.mark.gpu


def _cuda(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _done():
    torch.cuda.synchronize()
    la.get_device_error()


def test_decode_at_bench_size():
    w = W.Workload("decode", 64, 1, 32, 128, 128, torch.bfloat16, W.alibi_g_gamma(32),
                   128 ** -0.5, init_std=0.1)
    x = W.make_inputs(w, seed=11)
    d = _cuda(x)
    o, fin = la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], w.scale, d["initial_state"])
    _done()
    rows, heads = [0, 37, 63], [0, 13, 31]
    y = take_heads(x, heads, rows)
    ro, rf = oracle.forward(y["q"], y["k"], y["v"], y["g_gamma"], w.scale, y["initial_state"])
    compare(take_out(dict(o=o.cpu(), final_state=fin.cpu()), heads, rows),
            dict(o=ro, final_state=rf), TOL[torch.bfloat16], label="decode b64 h32 T1")


def test_sequence_split_at_bench_size():
    w = W.Workload("split", 1, 262144, 8, 128, 128, torch.bfloat16, W.alibi_g_gamma(8), 1.0,
                   dfinal_std=0.0)
    x = W.make_inputs(w, seed=13)
    d = _cuda(x)
    o, fin = la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], 1.0)
    dq, dk, dv, _ = la.la_bwd(d["q"], d["k"], d["v"], d["do"], d["g_gamma"], 1.0,
                              want_d_initial_state=False)
    _done()
    del d
    heads = [0, 7]
    y = take_heads(x, heads)
    ro, rf = oracle.forward(y["q"], y["k"], y["v"], y["g_gamma"], 1.0)
    rq, rk, rv, _ = oracle.backward(y["q"], y["k"], y["v"], y["g_gamma"], 1.0, y["do"])
    got = take_out(dict(o=o.cpu(), final_state=fin.cpu(), dq=dq.cpu(), dk=dk.cpu(),
                        dv=dv.cpu()), heads)
    compare(got, dict(o=ro, final_state=rf, dq=rq, dk=rk, dv=rv), TOL[torch.bfloat16],
            label="split b1 h8 n262144")


def test_grouped_heads_at_bench_size():
    B, T, H, Hkv, D = 4, 32768, 32, 8, 128
    G = H // Hkv
    w = W.Workload("gqa", B, T, H, D, D, torch.bfloat16, W.alibi_g_gamma(H), 1.0)
    x = W.make_inputs(w, seed=17)
    x["k"] = x["k"][:, :, ::G].contiguous()
    x["v"] = x["v"][:, :, ::G].contiguous()
    d = _cuda(x)
    o, fin = la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], 1.0)
    dq, dk, dv, _ = la.la_bwd(d["q"], d["k"], d["v"], d["do"], d["g_gamma"], 1.0,
                              want_d_initial_state=False)
    _done()
    del d
    # batch row 2, key/value head 5 and its query heads 20..23
    row, kvh = 2, 5
    qh = list(range(kvh * G, kvh * G + G))
    y = {"q": x["q"][row:row + 1, :, qh].contiguous(), "do": x["do"][row:row + 1, :, qh].contiguous(),
         "k": x["k"][row:row + 1, :, [kvh] * G].contiguous(),
         "v": x["v"][row:row + 1, :, [kvh] * G].contiguous(),
         "g_gamma": x["g_gamma"][qh].contiguous()}
    ro, rf = oracle.forward(y["q"], y["k"], y["v"], y["g_gamma"], 1.0)
    rq, rk, rv, _ = oracle.backward(y["q"], y["k"], y["v"], y["g_gamma"], 1.0, y["do"])
    got = dict(o=o[row:row + 1, :, qh].cpu(), final_state=fin[row:row + 1, qh].cpu(),
               dq=dq[row:row + 1, :, qh].cpu(), dk=dk[row:row + 1, :, kvh:kvh + 1].cpu(),
               dv=dv[row:row + 1, :, kvh:kvh + 1].cpu())
    ref = dict(o=ro, final_state=rf, dq=rq,
               dk=torch.as_tensor(rk).sum(2, keepdim=True), dv=torch.as_tensor(rv).sum(2, keepdim=True))
    compare(got, ref, TOL[torch.bfloat16], label="grouped b4 h32 kv8 n32768")


def test_gated_at_bench_size():
    B, T, H, D = 4, 8192, 32, 128
    w = W.Workload("gla", B, T, H, D, D, torch.bfloat16, W.alibi_g_gamma(H), 1.0,
                   dfinal_std=0.0)
    x = W.make_inputs(w, seed=19)
    gen = torch.Generator().manual_seed(1019)
    x["g"] = -0.3 * torch.rand(x["q"].shape, generator=gen)
    d = _cuda(x)
    o, fin, ops = la.gla_fwd(d["q"], d["k"], d["v"], d["g"], d["g_gamma"], 1.0,
                             keep_operands=True)
    assert ops is not None   # the chunked form ran
    dq, dk, dv, dg, _ = la.gla_bwd(d["q"], d["k"], d["v"], d["do"], d["g"], d["g_gamma"], 1.0,
                                   want_d_initial_state=False, operands=ops)
    _done()
    del d
    rows, heads = [0, 3], [0, 31]
    y = take_heads(x, heads, rows)
    y["g"] = x["g"][rows][:, :, heads].contiguous()
    ro, rf = oracle.gla_forward(y["q"], y["k"], y["v"], y["g"], y["g_gamma"], 1.0)
    rq, rk, rv, rg, _ = oracle.gla_backward(y["q"], y["k"], y["v"], y["g"], y["g_gamma"], 1.0,
                                            y["do"])
    got = take_out(dict(o=o.cpu(), final_state=fin.cpu(), dq=dq.cpu(), dk=dk.cpu(),
                        dv=dv.cpu(), dg=dg.cpu()), heads, rows)
    y["initial_state"] = y["d_final_state"] = None
    compare_gated(got, dict(o=ro, final_state=rf, dq=rq, dk=rk, dv=rv, dg=rg), y, False,
                  TOL[torch.bfloat16], "gated b4 h32 n8192")
