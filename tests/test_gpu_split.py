"""Sequence split: few (sequence, head) pairs, long sequences.

The library cuts long sequences into segments that run in parallel, in two
passes around a scan of one state per (segment, head).  These tests make it
engage on small problems (shortest segment 256 tokens), check forward and
backward against the oracle with initial and final-state gradients, in both
directions, for dense batches, packed sequences (one shorter than a segment,
one empty) and fp32 tokens, and check that a layout the split cannot view as
one row of tokens runs unsplit.
"""
import ctypes
import math

import pytest
import torch

import workloads as W
from linear_attention_head_gb300 import _native as N
from parity import TOL, compare, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def short_segments():
    N.check(N.lib().la_set_sequence_split(1, 256))
    yield
    N.check(N.lib().la_set_sequence_split(1, 0))


def _w(B, T, H, D, dtype, seqlens=None):
    return W.Workload("split", B, T if seqlens is None else sum(seqlens), H, D, D, dtype,
                      torch.tensor([-0.002, -0.3][:H] + [-0.01] * max(0, H - 2)),
                      1.0 / math.sqrt(D), seqlens=seqlens, init_std=0.2, dfinal_std=0.2)


def _ws_bytes(x, packed_n=0):
    d = N.LaDims()
    B, T, H, D = x["q"].shape
    E = x["v"].shape[3]
    d.batch, d.seq_len, d.heads, d.dim_qk, d.dim_v, d.num_seqs = B, T, H, D, E, packed_n
    for i in range(3):
        d.qk_strides[i] = x["q"].stride(i)
        d.v_strides[i] = x["v"].stride(i)
    code = N.LA_DTYPE_BF16 if x["q"].dtype == torch.bfloat16 else N.LA_DTYPE_F32
    cu = x["cu_seqlens"]
    keep = None if cu is None else cu.to(torch.int32).contiguous()
    host = None if keep is None else ctypes.c_void_p(keep.data_ptr())
    return int(N.lib().la_workspace_size_for(ctypes.byref(d), code, host))


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_dense_split_matches_oracle(dtype, D):
    x = W.make_inputs(_w(1, 5000, 2, D, dtype), seed=3)
    assert _ws_bytes(x) > 0            # the split engages for this call
    for reverse in (False, True):
        compare(gpu_run(x, reverse), oracle_run(x, reverse), TOL[dtype],
                label="split rev=%d" % reverse)


def test_packed_split_matches_oracle():
    lens = [3000, 17, 0, 2100, 700]
    x = W.make_inputs(_w(1, 0, 2, 128, torch.bfloat16, seqlens=lens), seed=4)
    assert _ws_bytes(x, len(lens)) > int(N.lib().la_workspace_size(len(lens)))
    for reverse in (False, True):
        got = gpu_run(x, reverse)
        compare(got, oracle_run(x, reverse), TOL[torch.bfloat16], cu=x["cu_seqlens"],
                label="packed split rev=%d" % reverse)
        # the empty sequence passes its states through
        assert torch.equal(got["final_state"][2], x["initial_state"][2])
        assert torch.equal(got["d_initial_state"][2], x["d_final_state"][2])


def test_split_and_unsplit_agree():
    x = W.make_inputs(_w(2, 4096, 2, 128, torch.bfloat16), seed=5)
    split = gpu_run(x)
    N.check(N.lib().la_set_sequence_split(0, 256))
    whole = gpu_run(x)
    for name in whole:
        a, b = split[name].float(), whole[name].float()
        assert (a - b).abs().max() <= 2e-2 * b.abs().max(), name


def test_layout_without_a_flat_token_view_runs_unsplit():
    # head-major [B, H, T, D]: a batch row is not T token strides long
    x = W.make_inputs(_w(2, 3000, 2, 128, torch.bfloat16), seed=6)
    for key in ("q", "k", "v", "do"):
        x[key] = x[key].transpose(1, 2).contiguous().transpose(1, 2)
    assert _ws_bytes(x) == 0
    compare(gpu_run(x), oracle_run(x), TOL[torch.bfloat16], label="head-major")


def test_long_single_sequence_few_heads():
    # one sequence, one head: the split's main case (25 segments of 384 tokens)
    x = W.make_inputs(_w(1, 9400, 1, 128, torch.bfloat16), seed=7)
    assert _ws_bytes(x) > 0
    compare(gpu_run(x), oracle_run(x), TOL[torch.bfloat16], label="b1 h1")
