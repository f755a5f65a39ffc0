"""Bounded on-device waits: every mbarrier wait of the tensor-core kernels gives
up after about 2 s, raises LA_ERR_TIMEOUT in a device word and returns, so an
error reaches the host instead of a hung GPU.  The test withholds one hand-off
inside the kernel (la_debug_withhold_next_handoff), so a wait is made to run
out; no fault, trap or endless loop is involved.  Afterwards the context must
still work: the same call without the switch matches the oracle."""
import time

import pytest
import torch

import linear_attention_head_gb300 as la
import workloads as W
from linear_attention_head_gb300 import _native as N
from parity import TOL, compare, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


def test_withheld_handoff_reports_timeout_and_context_survives():
    w = W.Workload("tiny_tc", 1, 300, 2, 128, 128, torch.bfloat16, W.alibi_g_gamma(2), 0.1,
                   backward=False)
    x = W.make_inputs(w, seed=51)
    assert la.kernel_family(1, 300, 2, 128, 128) == 1
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    la.get_device_error()                       # start from a clear word
    N.check(N.lib().la_debug_withhold_next_handoff(1))
    t0 = time.time()
    la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], w.scale)
    with pytest.raises(N.LaError) as err:
        la.get_device_error()
    assert err.value.status == N.LA_ERR_TIMEOUT
    assert time.time() - t0 < 60
    la.get_device_error()                       # the word was cleared by the read
    # the switch reset itself; the context still computes correctly
    got = gpu_run(x, backward=False)
    compare(got, oracle_run(x, backward=False), TOL[torch.bfloat16], label="after timeout")


@pytest.mark.parametrize("T", [1, 16])
def test_withheld_copy_in_streamed_decode_reports_timeout(T):
    # 20 x 16 = 320 (sequence, head) blocks of one token (the streamed decode
    # kernel, token by token) or 16 (its tensor-core form): the copy warp
    # then skips each CTA's first state block, so the compute warps' bounded
    # wait on it runs out
    assert torch.cuda.get_device_properties(0).multi_processor_count <= 160
    w = W.Workload("decode", 20, T, 16, 128, 128, torch.bfloat16, W.alibi_g_gamma(16), 0.1,
                   init_std=0.1, backward=False)
    x = W.make_inputs(w, seed=52)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    la.get_device_error()
    N.check(N.lib().la_debug_withhold_next_handoff(1))
    t0 = time.time()
    la.la_fwd(d["q"], d["k"], d["v"], d["g_gamma"], w.scale, d["initial_state"])
    with pytest.raises(N.LaError) as err:
        la.get_device_error()
    assert err.value.status == N.LA_ERR_TIMEOUT
    assert time.time() - t0 < 60
    la.get_device_error()
    got = gpu_run(x, backward=False)
    compare(got, oracle_run(x, backward=False), TOL[torch.bfloat16], label="after decode timeout")
