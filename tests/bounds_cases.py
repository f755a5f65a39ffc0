"""Runs small cases through the library named by LA_LIBRARY (the bounds-checking
build) and checks that no index check fired: every case that the oracle can
check is also compared with it at the parity tolerances.  Started by
tests/test_gpu_bounds_checked.py in a process of its own, so that the other
tests keep the normal library.  Exits 0 when all cases pass."""
import math
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import torch  # noqa: E402

import linear_attention_head_gb300 as la  # noqa: E402
import workloads as W  # noqa: E402
from linear_attention_head_gb300 import _native as N  # noqa: E402
from parity import TOL, compare, gpu_run, oracle_run  # noqa: E402


def custom(B, T, H, D, E, seqlens=None, init=0.1, dfin=0.1, g=None):
    g = W.alibi_g_gamma(H) if g is None else g
    return W.Workload("bounds", B, T if seqlens is None else sum(seqlens), H, D, E,
                      torch.bfloat16, g, 1.0 / math.sqrt(D), seqlens=seqlens, init_std=init,
                      dfinal_std=dfin)


def parity_case(label, w, seed):
    x = W.make_inputs(w, seed=seed)
    for reverse in (False, True):
        got = gpu_run(x, reverse)            # raises LaError(LA_ERR_BOUNDS) on a failed check
        compare(got, oracle_run(x, reverse), TOL[torch.bfloat16], cu=x["cu_seqlens"],
                label="%s rev=%d" % (label, reverse))


def main():
    assert N.lib().la_build_flags() & N.LA_BUILD_BOUNDS_CHECKED, "not the checked build"
    la.get_device_error()
    # d = e = 128: the sweep kernel and the fused dk/dv kernel; ragged tails,
    # packed sequences with empty and short ones, states in and out
    parity_case("dense d128", custom(2, 300, 2, 128, 128, g=torch.tensor([0.0, -0.7])), 1)
    parity_case("packed d128", custom(1, 0, 3, 128, 128, seqlens=[0, 1, 130, 0, 64, 257, 3, 128,
                                                                  129]), 2)
    # other widths: padded key blocks, state pieces, value tiles
    for D, E in ((64, 64), (192, 192), (256, 64), (64, 256), (128, 64), (128, 192)):
        parity_case("d%d e%d" % (D, E), custom(1, 0, 2, D, E, seqlens=[200, 0, 77]), D + E)
    # the sequence split: state-only first pass, scan, fused second pass
    N.check(N.lib().la_set_sequence_split(1, 128))
    try:
        parity_case("split d128", custom(1, 1100, 1, 128, 128), 3)
    finally:
        N.check(N.lib().la_set_sequence_split(1, 0))
    # grouped key/value heads (per-query-head contributions) and the gated
    # form on the tensor cores: run only, the index checks are what is read
    dev = "cuda"
    gen = torch.Generator(device=dev).manual_seed(5)
    B, T, H, Hkv, D = 1, 300, 4, 2, 128
    q, do = (torch.randn((B, T, H, D), generator=gen, device=dev).bfloat16() for _ in range(2))
    k, v = (torch.randn((B, T, Hkv, D), generator=gen, device=dev).bfloat16() for _ in range(2))
    g = W.alibi_g_gamma(H).to(dev)
    la.la_fwd(q, k, v, g, 0.1)
    la.la_bwd(q, k, v, do, g, 0.1)
    k, v = (torch.randn((B, T, H, D), generator=gen, device=dev).bfloat16() for _ in range(2))
    gate = -0.3 * torch.rand((B, T, H, D), generator=gen, device=dev)
    o, fin, ops = la.gla_fwd(q, k, v, gate, g, 0.1, keep_operands=True)
    la.gla_bwd(q, k, v, do, gate, g, 0.1, operands=ops)
    torch.cuda.synchronize()
    la.get_device_error()
    print("bounds-checked cases ok")


if __name__ == "__main__":
    main()
