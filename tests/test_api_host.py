"""Argument checks of the Python entry points that run before any device work
(CPU tensors, no GPU): packed calls need one batch row and one initial state
per sequence; 3-D inputs need cu_seqlens; the gk / gv gates are refused."""
import pytest
import torch

import linear_attention_head_gb300 as la


def _qkv(B, T, H=2, D=8):
    x = torch.zeros(B, T, H, D)
    return x, x.clone(), x.clone()


def test_packed_calls_need_one_batch_row():
    q, k, v = _qkv(2, 6)
    cu = torch.tensor([0, 3, 6], dtype=torch.int32)
    for fn in (la.recurrent, la.recurrent_gla):
        with pytest.raises(ValueError, match="batch dimension must be 1"):
            fn(q, k, v, cu_seqlens=cu)
    with pytest.raises(ValueError, match="batch dimension must be 1"):
        la.lightning_attn(q, k, v, 0, 4, cu_seqlens=cu)


def test_packed_calls_need_one_state_per_sequence():
    q, k, v = _qkv(1, 6)
    cu = torch.tensor([0, 3, 6], dtype=torch.int32)
    s0 = torch.zeros(3, 2, 8, 8)
    with pytest.raises(ValueError, match="2 sequences, 3 states"):
        la.recurrent_gla(q, k, v, cu_seqlens=cu, initial_state=s0)
    with pytest.raises(ValueError, match="2 sequences, 3 states"):
        la.lightning_attn(q, k, v, 1, 4, cu_seqlens=cu, initial_state=s0)


def test_three_dim_inputs_need_cu_seqlens_and_extra_gates_are_refused():
    q, k, v = _qkv(1, 6)
    with pytest.raises(ValueError, match="cu_seqlens"):
        la.recurrent(q[0], k[0], v[0])
    with pytest.raises(NotImplementedError):
        la.recurrent(q, k, v, gk=torch.zeros(1))


def test_lightning_keys_take_the_queries_shape():
    q, k, v = _qkv(1, 6)
    with pytest.raises(ValueError, match="shape of query"):
        la.lightning_attn(q, k[:, :, :1], v, 0, 4)


def test_layer_dependent_decay():
    # g_gamma[h] = -(8/H)(1 - l/L) h: zero for head 0, steepest in the first layer
    g = la.lightning_g_gamma(8, 0, 4)
    assert g.dtype == torch.float32 and g.shape == (8,)
    assert g[0] == 0 and torch.allclose(g[1:] / g[1], torch.arange(1, 8, dtype=torch.float32))
    assert torch.isclose(g[1], torch.tensor(-1.0))
    assert torch.isclose(la.lightning_g_gamma(8, 2, 4)[1], torch.tensor(-0.5))


def test_alibi_decay():
    # head i of H decays by exp(-2^(-8 i / H)) per token: slopes halve every H/8 heads
    g = la.alibi_g_gamma(32)
    assert g.dtype == torch.float32 and g.shape == (32,)
    assert torch.all(g < 0) and torch.all(g[1:] > g[:-1])
    assert g[-1] == -2.0 ** -8 and g[3] == -0.5
    assert torch.allclose(g[4:] / g[:-4], torch.full((28,), 0.5))


def test_nvtx_ranges_are_opt_in():
    # without LA_NVTX the entry points are the plain functions; with LA_NVTX=1 they
    # are wrapped, and a call that fails validation still closes its range
    import os
    import subprocess
    import sys
    assert not hasattr(la.la_fwd, "__wrapped__")
    code = ("import torch, linear_attention_head_gb300 as la\n"
            "assert hasattr(la.la_fwd, '__wrapped__') and la.la_fwd.__name__ == 'la_fwd'\n"
            "try:\n"
            "    la.la_fwd(torch.zeros(1, 2, 1, 4), torch.zeros(1, 2, 1, 4),\n"
            "              torch.zeros(1, 2, 1, 4), torch.zeros(1))\n"
            "except ValueError:\n"
            "    print('raised')\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    run = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         cwd=root, env=dict(os.environ, LA_NVTX="1"), timeout=300)
    assert run.returncode == 0, run.stderr
    assert "raised" in run.stdout
