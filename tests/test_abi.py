"""Host-only checks of the C ABI (no GPU, no kernel launches).

* the library loads and exports every function include/la.h declares;
* the ctypes prototypes cover exactly those functions;
* every validation failure returns its status before anything touches CUDA
  (these calls would otherwise need a device), and la_last_error explains it;
* la_kernel_family and la_strerror are pure host functions.
"""
import ctypes
import os
import re
import subprocess

import pytest

import linear_attention_head_gb300 as la
from linear_attention_head_gb300 import _native as N
from linear_attention_head_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "la.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return N.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("la_fwd", "la_bwd", "la_bwd_dq", "la_bwd_dkdv", "la_strerror",
                 "la_last_error", "la_get_device_error", "la_kernel_family", "la_version"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", libbuild.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s+(la_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_prototypes_match_header():
    assert sorted(N.PROTOTYPES) == declared_functions()


def test_dims_struct_layout():
    # int32 x 6, two int64[3], int32 x 2, two int64[3]: no padding anywhere
    assert ctypes.sizeof(N.LaDims) == 128
    assert N.LaDims.qk_strides.offset == 24
    assert N.LaDims.v_strides.offset == 48
    assert N.LaDims.kv_heads.offset == 72
    assert N.LaDims.k_strides.offset == 80
    assert N.LaDims.kv_v_strides.offset == 104


def test_grouped_heads_are_validated(lib):
    d = _dims(H=4)
    d.kv_heads = 3                                   # does not divide 4
    assert _fwd(lib, d) == N.LA_ERR_INVALID_ARG
    assert "kv_heads" in N.last_error()
    d.kv_heads = 5
    assert _fwd(lib, d) == N.LA_ERR_INVALID_ARG
    d = _dims(H=4)
    d.reserved = 1
    assert _fwd(lib, d) == N.LA_ERR_INVALID_ARG
    d = _dims(H=4)
    d.kv_heads = 2
    d.k_strides[1] = -1
    assert _fwd(lib, d) == N.LA_ERR_INVALID_ARG


def test_strerror_and_version(lib):
    assert N.strerror(0) == "ok"
    assert "invalid" in N.strerror(1)
    assert N.strerror(99) == "unknown status"
    assert lib.la_version() >= 1


def _dims(B=2, T=16, H=2, D=64, E=64, N_=0, layout="bthd"):
    d = N.LaDims()
    d.batch, d.seq_len, d.heads, d.dim_qk, d.dim_v, d.num_seqs = B, T, H, D, E, N_
    qs = (T * H * D, H * D, D) if layout == "bthd" else (H * T * D, D, T * D)
    vs = (T * H * E, H * E, E) if layout == "bthd" else (H * T * E, E, T * E)
    for i in range(3):
        d.qk_strides[i], d.v_strides[i] = qs[i], vs[i]
    return d


FAKE = ctypes.c_void_p(0x1000)     # never dereferenced: validation fails first


def _fwd(lib, dims, dtype=0, cu=None, cu_host=None, q=FAKE, g=FAKE, o=FAKE):
    return lib.la_fwd(ctypes.byref(dims) if dims is not None else None, dtype, q, FAKE, FAKE, g,
                      1.0, None, 0, cu, cu_host, o, None, None, 0, None)


def test_validation_errors_return_before_any_launch(lib):
    assert _fwd(lib, None) == N.LA_ERR_INVALID_ARG
    assert "dims" in N.last_error()
    assert _fwd(lib, _dims(), dtype=7) == N.LA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(B=-1)) == N.LA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(H=0)) == N.LA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(D=0)) == N.LA_ERR_UNSUPPORTED
    assert _fwd(lib, _dims(E=300)) == N.LA_ERR_UNSUPPORTED
    assert _fwd(lib, _dims(), q=None) == N.LA_ERR_INVALID_ARG
    assert "q is NULL" in N.last_error()
    assert _fwd(lib, _dims(), o=None) == N.LA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(), g=None) == N.LA_ERR_INVALID_ARG
    d = _dims()
    d.qk_strides[1] = -1
    assert _fwd(lib, d) == N.LA_ERR_INVALID_ARG


def _cu(vals):
    arr = (ctypes.c_int32 * len(vals))(*vals)
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def test_packed_sequence_table_is_validated_on_the_host(lib):
    good, gp = _cu([0, 5, 5, 16])
    # batch must be 1 with cu_seqlens (lightning_attn docstring, Raises)
    assert _fwd(lib, _dims(B=2, N_=3), cu=FAKE, cu_host=gp) == N.LA_ERR_INVALID_ARG
    assert "batch must be 1" in N.last_error()
    bad0, b0 = _cu([1, 5, 5, 16])
    assert _fwd(lib, _dims(B=1, N_=3), cu=FAKE, cu_host=b0) == N.LA_ERR_INVALID_ARG
    dec, dp = _cu([0, 6, 5, 16])
    assert _fwd(lib, _dims(B=1, N_=3), cu=FAKE, cu_host=dp) == N.LA_ERR_INVALID_ARG
    assert "decreases" in N.last_error()
    last, lp = _cu([0, 5, 5, 15])
    assert _fwd(lib, _dims(B=1, N_=3), cu=FAKE, cu_host=lp) == N.LA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(B=1, N_=-1), cu=FAKE, cu_host=gp) == N.LA_ERR_INVALID_ARG
    # a host table without the device table is an error too
    assert _fwd(lib, _dims(B=1, N_=3), cu=None, cu_host=gp) == N.LA_ERR_INVALID_ARG


def test_backward_entry_points_validate(lib):
    d = _dims()
    st = lib.la_bwd(ctypes.byref(d), 0, FAKE, FAKE, FAKE, None, FAKE, 1.0, None, None, 0, None,
                    None, FAKE, FAKE, FAKE, None, None, 0, None)
    assert st == N.LA_ERR_INVALID_ARG and "d_o" in N.last_error()
    st = lib.la_bwd_dq(ctypes.byref(d), 0, None, FAKE, FAKE, FAKE, FAKE, 1.0, None, 0, None,
                       None, None, None, 0, None)
    assert st == N.LA_ERR_INVALID_ARG and "dq" in N.last_error()
    st = lib.la_bwd_dkdv(ctypes.byref(d), 0, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, None, 0, None,
                         None, FAKE, None, None, None, 0, None)
    assert st == N.LA_ERR_INVALID_ARG and "dv" in N.last_error()


def test_empty_problems_enqueue_nothing(lib):
    # zero batch rows or zero packed sequences: nothing to compute, success
    assert _fwd(lib, _dims(B=0), q=None, o=None) == N.LA_OK
    empty, ep = _cu([0])
    assert _fwd(lib, _dims(B=1, T=0, N_=0), cu=FAKE, cu_host=ep, q=None, o=None) == N.LA_OK


def test_kernel_family_is_host_only():
    assert la.kernel_family(4, 1024, 32, 128, 128) in (0, 1)
    assert la.kernel_family(1, 256, 2, 32, 32, dtype="f32") == 0
    assert la.kernel_family(1, 256, 2, 0, 32) == -1


def test_workspace_size(lib):
    assert lib.la_workspace_size(0) == 0
    assert lib.la_workspace_size(1) == 256
    assert lib.la_workspace_size(64) == 256
    assert lib.la_workspace_size(65) == 512


def test_split_planning_by_head_width(lib):
    # la_debug_split_segments plans for a given SM count without a device.
    # Automatic segments: >= 256 tokens at d <= 64, >= 4 segments of >= 1024
    # tokens at d <= 128, none above; only when the pairs fill at most half
    # of the SMs.
    seg = lambda d, sms=152: lib.la_debug_split_segments(ctypes.byref(d), 0, None, sms)
    assert lib.la_set_sequence_split(1, 0) == N.LA_OK
    assert seg(_dims(B=2, T=2048, H=8, D=64, E=64)) == 2 * 8        # 256-token segments
    assert seg(_dims(B=2, T=4096, H=16, D=128, E=128)) == 2 * 4     # 4 x 1024
    assert seg(_dims(B=2, T=2048, H=8, D=128, E=128)) == 0          # only 2 of 1024
    assert seg(_dims(B=2, T=2048, H=12, D=192, E=192)) == 0         # wide heads: never
    assert seg(_dims(B=1, T=262144, H=8, D=128, E=128)) == 19       # 152 / 8 pairs
    assert seg(_dims(B=4, T=32768, H=32, D=128, E=128)) == 0        # 128 pairs > 76
    assert seg(_dims(B=2, T=4096, H=16, D=128, E=128), sms=0) == -1
    # an explicit minimum applies at any width, from 2 segments
    assert lib.la_set_sequence_split(1, 256) == N.LA_OK
    try:
        assert seg(_dims(B=2, T=2048, H=8, D=128, E=128)) == 2 * 8
        d = _dims(B=1, T=5817, H=2, D=128, E=128, N_=5)
        _, cp = _cu([0, 3000, 3017, 3017, 5117, 5817])
        # R = min(152 / 10, 3000 / 256) = 11 -> 384-token segments: 8 + 1 + 0 + 6 + 2
        assert lib.la_debug_split_segments(ctypes.byref(d), 0, cp, 152) == 17
        assert lib.la_set_sequence_split(0, 0) == N.LA_OK
        assert seg(_dims(B=1, T=262144, H=8, D=128, E=128)) == 0
    finally:
        assert lib.la_set_sequence_split(1, 0) == N.LA_OK


def test_workspace_size_for_and_split_control(lib):
    # no device here: the split cannot be planned, only the packed schedule is sized
    d = _dims(B=1, T=16, N_=3)
    cu, cp = _cu([0, 5, 5, 16])
    assert lib.la_workspace_size_for(ctypes.byref(d), 0, cp) == lib.la_workspace_size(3)
    assert lib.la_workspace_size_for(ctypes.byref(_dims()), 0, None) == 0
    assert lib.la_workspace_size_for(ctypes.byref(_dims(H=0)), 0, None) == 0
    assert lib.la_set_sequence_split(2, 2048) == N.LA_ERR_INVALID_ARG
    assert lib.la_set_sequence_split(1, 64) == N.LA_ERR_INVALID_ARG
    assert lib.la_set_sequence_split(0, 4096) == N.LA_OK
    assert lib.la_set_sequence_split(1, 2048) == N.LA_OK
    assert lib.la_set_sequence_split(1, 127) == N.LA_ERR_INVALID_ARG
    assert lib.la_set_sequence_split(1, 0) == N.LA_OK   # automatic, the default


def test_gated_forward_workspace_size(lib):
    # the chunked gated forward applies to bf16, D = 128, E in {64, 128} and
    # sequences longer than 16 tokens: q~ and k~ (bf16), two fp32 vectors per
    # 128-token chunk and (sequence, head), one flag per (sequence, head)
    big = _dims(B=2, T=300, H=3, D=128, E=128)
    r = lambda x: (x + 255) // 256 * 256
    tok, vec = 2 * 300 * 3 * 128 * 2, 2 * 3 * 3 * 128 * 4
    assert lib.la_gla_fwd_workspace_size(ctypes.byref(big), 0, None) == \
        2 * r(tok) + 2 * r(vec) + r(2 * 3 * 4)
    assert lib.la_gla_fwd_workspace_size(ctypes.byref(big), 1, None) == 0
    assert lib.la_gla_fwd_workspace_size(ctypes.byref(_dims(T=16, D=128, E=128)), 0, None) == 0
    assert lib.la_gla_fwd_workspace_size(ctypes.byref(_dims(T=300, D=64)), 0, None) == 0
    assert lib.la_gla_fwd_workspace_size(ctypes.byref(_dims(T=300, D=128, E=64)), 0, None) > 0


def test_gated_backward_workspace_with_forward_operands(lib):
    # with the forward's operands the backward needs only its token-by-token
    # part; the difference is the forward's workspace where the chunked
    # backward applies (bf16, D = 128, E in {64, 128}), nothing otherwise
    for E in (128, 64):
        d = _dims(B=2, T=300, H=3, D=128, E=E)
        full = lib.la_gla_workspace_size(ctypes.byref(d), 0, None, 0)
        part = lib.la_gla_workspace_size(ctypes.byref(d), 0, None, 1)
        assert full - part == lib.la_gla_fwd_workspace_size(ctypes.byref(d), 0, None) > 0
    for d in (_dims(B=2, T=300, H=3, D=64, E=64), _dims(B=2, T=300, H=3, D=128, E=96)):
        assert lib.la_gla_workspace_size(ctypes.byref(d), 0, None, 0) == \
            lib.la_gla_workspace_size(ctypes.byref(d), 0, None, 1) > 0


def test_gated_backward_workspace_holds_fp32_gradients(lib):
    # the token-by-token part: the final state (fp32, transposed), dg's block
    # sums (fp32, one per 256 tokens, channel and (sequence, head)) and, for
    # bf16 tokens, dq and dk in fp32 ([B][T][H][D]), which dg takes unrounded
    r = lambda x: (x + 255) // 256 * 256
    d = _dims(B=2, T=300, H=3, D=128, E=96)
    state, bsum, tokf = 2 * 3 * 128 * 96 * 4, 2 * 3 * 2 * 128 * 4, 2 * 300 * 3 * 128 * 4
    assert lib.la_gla_workspace_size(ctypes.byref(d), 1, None, 1) == r(state) + r(bsum)
    assert lib.la_gla_workspace_size(ctypes.byref(d), 0, None, 1) == \
        r(state) + r(bsum) + 2 * r(tokf)


def test_gated_backward_workspace_with_grouped_heads(lib):
    # grouped key/value heads: every query head's part of dk in the fp32 rows
    # (also for fp32 tokens, where dq and dk otherwise go straight to the
    # caller) and of dv ([B][T][H][E], token dtype), summed per group at the end
    r = lambda x: (x + 255) // 256 * 256
    B, T, H, Hkv, D, E = 2, 300, 6, 2, 128, 96
    d = _dims(B=B, T=T, H=H, D=D, E=E)
    d.kv_heads = Hkv
    for i, (ks, vs) in enumerate(zip((T * Hkv * D, Hkv * D, D), (T * Hkv * E, Hkv * E, E))):
        d.k_strides[i], d.kv_v_strides[i] = ks, vs
    state, bsum, tokf = B * H * D * E * 4, B * H * 2 * D * 4, B * T * H * D * 4
    for dtype, esz in ((0, 2), (1, 4)):
        assert lib.la_gla_workspace_size(ctypes.byref(d), dtype, None, 1) == \
            r(state) + r(bsum) + 2 * r(tokf) + r(B * T * H * E * esz)
    # the same sizes with kv_heads = heads: k's own strides, no group sums
    d1 = _dims(B=B, T=T, H=H, D=D, E=E)
    d1.kv_heads = H
    for i, (ks, vs) in enumerate(zip((T * H * D, H * D, D), (T * H * E, H * E, E))):
        d1.k_strides[i], d1.kv_v_strides[i] = ks, vs
    assert lib.la_gla_workspace_size(ctypes.byref(d1), 1, None, 1) == r(state) + r(bsum)
    d1.k_strides[1] = H * D + 8     # k strided unlike q: the fp32 rows again
    d1.k_strides[0] = T * (H * D + 8)
    assert lib.la_gla_workspace_size(ctypes.byref(d1), 1, None, 1) == \
        r(state) + r(bsum) + 2 * r(tokf)
