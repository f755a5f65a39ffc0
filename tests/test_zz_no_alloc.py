"""la_fwd_noalloc: the forward pass for callers that cannot allocate device memory
at the point of the call (for instance because another allocator owns all of
the device's memory, or because a cudaMalloc there would synchronize the
device).  It keeps the packed-sequence schedule in an array compiled into the
library instead of a caller workspace.

The test calls it through the C ABI and compares its output with la_fwd's on
two calls in a row (the array keeps the previous call's schedule, so the
second call must not depend on leftovers).  Both entry points run the same
kernels on the same longest-first schedule (la_fwd is given a workspace of
exactly the schedule's size, as la_fwd_noalloc passes on), so the outputs
must be identical bit for bit, which is stricter than the parity tolerance.
The dense-batch case does not touch the array (there is no schedule without
cu_seqlens); it checks that the entry point passes dense calls through.
It also checks that more packed sequences than the array holds are rejected
before anything runs.  It builds all of its inputs itself, so it passes alone
in a fresh process as well as after the other tests.  This file is collected
last on purpose.
"""
import ctypes

import pytest
import torch

import workloads as W
from linear_attention_head_gb300 import _native as N

pytestmark = pytest.mark.gpu


def _dims(q, v, num_seqs):
    d = N.LaDims()
    d.batch, d.seq_len, d.heads, d.dim_qk, d.dim_v = q.shape[0], q.shape[1], q.shape[2], \
        q.shape[3], v.shape[3]
    d.num_seqs = num_seqs
    for i in range(3):
        d.qk_strides[i] = q.stride(i)
        d.v_strides[i] = v.stride(i)
    return d


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _run(entry, x, reverse):
    """One forward call through the C ABI; returns (o, final_state) on the host."""
    lib = N.lib()
    q, k, v, g = (x[n].cuda() for n in ("q", "k", "v", "g_gamma"))
    init = x["initial_state"].cuda() if x["initial_state"] is not None else None
    cu_host = x["cu_seqlens"]
    cu_dev = cu_host.cuda() if cu_host is not None else None
    n_seq = cu_host.numel() - 1 if cu_host is not None else q.shape[0]
    o = torch.full_like(v, float("nan"))
    fin = torch.full((n_seq, q.shape[2], q.shape[3], v.shape[3]), float("nan"),
                     device="cuda", dtype=torch.float32)
    dims = _dims(q, v, n_seq if cu_host is not None else 0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    common = [ctypes.byref(dims), N.LA_DTYPE_BF16 if q.dtype == torch.bfloat16 else N.LA_DTYPE_F32,
              _p(q), _p(k), _p(v), _p(g), float(x["scale"]), _p(init), int(reverse),
              _p(cu_dev), _p(cu_host), _p(o), _p(fin)]
    if entry == "la_fwd":
        ws = None
        nbytes = int(lib.la_workspace_size(n_seq)) if cu_host is not None else 0
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        st = lib.la_fwd(*common, _p(ws), nbytes, stream)
    else:
        st = lib.la_fwd_noalloc(*common, stream)
    N.check(st)
    torch.cuda.synchronize()
    return o.cpu(), fin.cpu()


def _packed(seed, lens, D, dtype=torch.bfloat16):
    w = W.Workload("packed", 1, sum(lens), 3, D, D, dtype, W.alibi_g_gamma(3), D ** -0.5,
                   seqlens=lens, init_std=0.1, backward=False)
    return W.make_inputs(w, seed=seed)


@pytest.mark.parametrize("D", [128, 64])
def test_no_alloc_forward_matches_la_fwd_on_two_calls(D):
    # two different packed batches in a row: the second call's schedule replaces
    # the first's in the shared array
    first = _packed(41, [300, 5, 0, 1000, 129, 64, 7], D)
    second = _packed(42, [17, 2000, 128, 3], D)
    for x, reverse in ((first, False), (second, True)):
        o_ref, f_ref = _run("la_fwd", x, reverse)
        o, f = _run("la_fwd_noalloc", x, reverse)
        assert not torch.isnan(o).any() and not torch.isnan(f).any()
        assert torch.equal(o, o_ref)
        assert torch.equal(f, f_ref)


def test_no_alloc_forward_dense_batch_matches_la_fwd():
    w = W.sweep_bf16(512)
    x = W.make_inputs(w, seed=43)
    x["do"] = None
    o_ref, f_ref = _run("la_fwd", x, False)
    o, f = _run("la_fwd_noalloc", x, False)
    assert torch.equal(o, o_ref)
    assert torch.equal(f, f_ref)


def test_no_alloc_forward_rejects_too_many_sequences():
    lib = N.lib()
    n_seq = N.LA_FWD_NOALLOC_MAX_SEQS + 1
    cu = torch.arange(n_seq + 1, dtype=torch.int32)          # one token per sequence
    q = torch.zeros((1, n_seq, 1, 64), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(1, device="cuda")
    dims = _dims(q, q, n_seq)
    st = lib.la_fwd_noalloc(ctypes.byref(dims), N.LA_DTYPE_BF16, _p(q), _p(q), _p(q), _p(g), 1.0,
                            None, 0, _p(cu.cuda()), _p(cu), _p(q.clone()), None,
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == N.LA_ERR_UNSUPPORTED
    assert "at most %d" % N.LA_FWD_NOALLOC_MAX_SEQS in N.last_error()
