"""Short sequences (at most 16 tokens): the token-by-token kernels.

Decoding a few new tokens against a carried state is the serving use of the
recurrence (the pages' `recurrent` API, an initial state in and the final
state out).  These calls run la_token.cu instead of the chunked kernels; the
tests check them against the oracle at every flag, head width and dtype, and
check that decoding a sequence piece by piece, each call's final state fed to
the next as its initial state, equals one call over the whole sequence.
"""
import math

import pytest
import torch

import linear_attention_head_gb300 as la
import workloads as W
from parity import TOL, compare, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


def _w(B, T, H, D, E, dtype, seqlens=None, g=None, init=0.3, dfin=0.3):
    g = W.alibi_g_gamma(H) if g is None else g
    return W.Workload("short", B, T if seqlens is None else sum(seqlens), H, D, E, dtype, g,
                      1.0 / math.sqrt(D), seqlens=seqlens, init_std=init, dfinal_std=dfin)


def test_kernel_family_switches_at_16_tokens():
    assert la.kernel_family(4, 1, 32, 128, 128) == 2
    assert la.kernel_family(4, 16, 32, 128, 128) == 2
    assert la.kernel_family(4, 17, 32, 128, 128) == 1
    assert la.kernel_family(1, 8, 2, 64, 48, dtype=torch.float32) == 2


@pytest.mark.parametrize("T", [1, 2, 7, 16])
@pytest.mark.parametrize("dtype,D,E", [(torch.bfloat16, 128, 128), (torch.bfloat16, 128, 16),
                                       (torch.float32, 64, 64),
                                       (torch.bfloat16, 192, 192), (torch.bfloat16, 16, 48),
                                       (torch.float32, 1, 1), (torch.bfloat16, 256, 40)])
def test_short_matches_oracle(T, dtype, D, E):
    w = _w(2, T, 3, D, E, dtype, g=torch.tensor([0.0, -0.05, -2.0]))
    x = W.make_inputs(w, seed=100 + T)
    for reverse in (False, True):
        compare(gpu_run(x, reverse), oracle_run(x, reverse), TOL[dtype],
                label="T=%d D=%d E=%d rev=%d" % (T, D, E, reverse))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_short_packed_with_empty_sequences(dtype):
    lens = [1, 0, 16, 5, 0, 11, 2]
    w = _w(1, 0, 4, 128, 128, dtype, seqlens=lens, init=0.1, dfin=0.1)
    x = W.make_inputs(w, seed=9)
    for reverse in (False, True):
        got = gpu_run(x, reverse)
        compare(got, oracle_run(x, reverse), TOL[dtype], cu=x["cu_seqlens"],
                label="packed short rev=%d" % reverse)
        for n in (1, 4):   # zero-length sequences pass their states through
            assert torch.equal(got["final_state"][n], x["initial_state"][n])
            assert torch.equal(got["d_initial_state"][n], x["d_final_state"][n])


def test_decoding_piece_by_piece_equals_one_call():
    # a 160-token sequence: one call (chunked kernels), or pieces of 1..16
    # tokens (token-by-token kernels) chained through the state, and one
    # longer piece (chunked kernels)
    B, T, H, D = 2, 160, 4, 128
    w = _w(B, T, H, D, D, torch.bfloat16, init=0.2, dfin=0.0)
    x = W.make_inputs(w, seed=21)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o_all, s_all = la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], w.scale, d["initial_state"])
    pieces, t, state, outs = [1, 1, 7, 16, 15, 16, 1, 16, 87], 0, d["initial_state"], []
    assert sum(pieces) == T
    for p in pieces:
        sl = slice(t, t + p)
        o, state = la.la_fwd(d["q"][:, sl], d["k"][:, sl], d["v"][:, sl], d["g_gamma"], w.scale,
                             state)
        outs.append(o)
        t += p
    torch.cuda.synchronize()
    la.get_device_error()
    o_dec = torch.cat(outs, dim=1)
    ref = oracle_run(x, backward=False)
    compare(dict(o=o_dec.cpu(), final_state=state.cpu()), ref, TOL[torch.bfloat16],
            label="decoded")
    compare(dict(o=o_all.cpu(), final_state=s_all.cpu()), ref, TOL[torch.bfloat16],
            label="one call")


# At least twice as many (sequence, head) blocks as the GPU has SMs: the
# streamed decode kernel (state blocks moved through shared memory by bulk
# copies) runs calls of at most 4 tokens token by token, and of 5 to 16
# tokens (key width a multiple of 8) as one chunk of the chunked form: one
# group of 8 tokens or two, every row-group count (D = 8..256); D = 12 takes
# the per-CTA kernel.  bf16 with D = 128 and E a multiple of 16 runs 5 to 16
# tokens on the tensor cores instead (la_decode.cu: its streamed form at
# E = 128, its per-CTA form at E = 48), E = 40 not.  20 x 16 = 320 blocks
# covers GPUs of up to 160 SMs.
@pytest.mark.parametrize("T", [1, 4, 5, 9, 16])
@pytest.mark.parametrize("dtype,D,E", [(torch.bfloat16, 128, 128), (torch.float32, 64, 64),
                                       (torch.bfloat16, 32, 96), (torch.bfloat16, 48, 80),
                                       (torch.bfloat16, 256, 64), (torch.float32, 16, 128),
                                       (torch.bfloat16, 8, 32), (torch.float32, 12, 20),
                                       (torch.bfloat16, 128, 48), (torch.bfloat16, 128, 40),
                                       (torch.bfloat16, 128, 64)])
@pytest.mark.parametrize("init", [0.3, 0.0])
def test_streamed_decode_matches_oracle(T, dtype, D, E, init):
    assert torch.cuda.get_device_properties(0).multi_processor_count <= 160
    w = _w(20, T, 16, D, E, dtype, init=init, dfin=0.0)
    x = W.make_inputs(w, seed=300 + T + D)
    for reverse in (False, True):
        compare(gpu_run(x, reverse, backward=False), oracle_run(x, reverse, backward=False),
                TOL[dtype], label="streamed T=%d D=%d E=%d init=%g rev=%d" % (T, D, E, init,
                                                                                 reverse))


@pytest.mark.parametrize("longest", [4, 16])
def test_streamed_decode_packed_and_in_place(longest):
    # 330 packed sequences of 0..4 tokens (the streamed kernel, token by
    # token) or 0..16 (as chunks); the state updated in place (initial and
    # final state the same buffer)
    gen = torch.Generator().manual_seed(5)
    lens = torch.randint(0, longest + 1, (330,), generator=gen).tolist()
    w = _w(1, 0, 2, 128, 128, torch.bfloat16, seqlens=lens, init=0.2, dfin=0.0)
    x = W.make_inputs(w, seed=12)
    ref = oracle_run(x, backward=False)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    state = d["initial_state"].clone()
    o, fin = la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], w.scale, state,
                       cu_seqlens=x["cu_seqlens"], final_state=state)
    torch.cuda.synchronize()
    la.get_device_error()
    assert fin.data_ptr() == state.data_ptr()
    compare(dict(o=o.cpu(), final_state=fin.cpu()), ref, TOL[torch.bfloat16],
            cu=x["cu_seqlens"], label="streamed packed in place")
