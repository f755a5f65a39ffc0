"""Tensor-level API over the C ABI: argument marshalling only.

Every step of the computation runs in the CUDA kernels of liblagb300.so; this
module only checks devices/dtypes, allocates outputs with torch (device
memory), and passes pointers, strides and the current CUDA stream.

Entry points mirror the pages:
  * `la_fwd` / `la_bwd` / `la_bwd_dq` / `la_bwd_dkdv`: the C ABI, one call each.
  * `recurrent(query, key, value, g_gamma=..., ...)`: ejkernel's `recurrent`
    restricted to the Lightning `g_gamma` gate, differentiable.
  * `lightning_attn(query, key, value, layer_idx, num_layers, ...)`: ejkernel's
    Lightning wrapper (layer-dependent g_gamma).
  * `lightning_attn_func(q, k, v, s)`: the Lightning-Attention-2 README call,
    layout (b, h, n, d), decay exp(-s).
"""
from __future__ import annotations

import ctypes
import functools
import math
import os
from typing import Optional, Tuple

import torch

from . import _native as N

Tensor = torch.Tensor

# LA_NVTX=1 in the environment when the package is imported: every C-ABI entry
# point below runs inside an NVTX range named after it (for Nsight Systems or
# `ncu --nvtx`).  Otherwise the functions are left as they are.
_NVTX = os.environ.get("LA_NVTX", "0") not in ("", "0")


def _traced(fn):
    if not _NVTX:
        return fn

    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        torch.cuda.nvtx.range_push(fn.__name__)
        try:
            return fn(*args, **kwargs)
        finally:
            torch.cuda.nvtx.range_pop()
    return wrapper


def lightning_g_gamma(num_heads: int, layer_idx: int, num_layers: int) -> Tensor:
    """The layer-dependent decay of the ejkernel lightning_attn page (module
    docstring): head h of layer l out of L gets g_gamma[h] = -(8/H)(1 - l/L) h."""
    return -(8.0 / num_heads * (1.0 - layer_idx / num_layers)) * torch.arange(
        num_heads, dtype=torch.float32)


def alibi_g_gamma(num_heads: int) -> Tensor:
    """Per-head log-decay from ALiBi-style slopes: g_gamma[i-1] = -2^(-8 i / H),
    i = 1..H, so head i decays by exp(-slope_i) per token.  The Lightning-Attention
    README's usage section builds such a slope tensor for its decay; the list is
    not printed there, and this is the geometric ALiBi recipe."""
    i = torch.arange(1, num_heads + 1, dtype=torch.float64)
    return (-(2.0 ** (-8.0 * i / num_heads))).to(torch.float32)


def _dtype_code(t: Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return N.LA_DTYPE_BF16
    if t.dtype == torch.float32:
        return N.LA_DTYPE_F32
    raise TypeError("token tensors must be bfloat16 or float32, got %s" % t.dtype)


def _ptr(t: Optional[Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


class _Packed:
    """cu_seqlens on the device plus a host copy (so the library never syncs), and the
    device workspace the library asks for (la_workspace_size_for: the longest-first
    schedule of packed sequences and the sequence split)."""

    def __init__(self, cu_seqlens, device):
        self.dev = None
        self.host = None
        self.n = 0
        self.ws = None
        self.device = device
        if cu_seqlens is None:
            return
        cu = torch.as_tensor(cu_seqlens)
        if cu.ndim != 1:
            raise ValueError("cu_seqlens must be 1-D")
        self.host = cu.detach().to("cpu", torch.int32).contiguous()
        if cu.device.type == "cuda" and cu.dtype == torch.int32 and cu.is_contiguous():
            self.dev = cu
        else:
            self.dev = self.host.to(device)
        self.n = self.host.numel() - 1

    def ws_args(self, dims, dtype_code):
        nbytes = int(N.lib().la_workspace_size_for(ctypes.byref(dims), dtype_code,
                                                   self.host_ptr()))
        if nbytes == 0:
            return None, 0
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return ctypes.c_void_p(self.ws.data_ptr()), nbytes

    def host_ptr(self):
        return None if self.host is None else ctypes.c_void_p(self.host.data_ptr())


def _check_tokens(q, k, v, extra=()):
    """q [B,T,H,D]; k [B,T,H_kv,D] and v [B,T,H_kv,E] with H_kv dividing H (grouped
    key/value heads, ejkernel `recurrent`'s num_kv_heads)."""
    ok = (q.ndim == 4 and k.ndim == 4 and v.ndim == 4 and k.shape[:2] == q.shape[:2]
          and k.shape[3] == q.shape[3] and v.shape[:3] == k.shape[:3] and k.shape[2] >= 1
          and q.shape[2] % k.shape[2] == 0)
    if not ok:
        raise ValueError("q must be [B, T, H, D], k [B, T, H_kv, D] and v [B, T, H_kv, E] "
                         "with H_kv dividing H (got %s, %s, %s)"
                         % (tuple(q.shape), tuple(k.shape), tuple(v.shape)))
    for t in (q, k, v) + tuple(extra):
        if t.device.type != "cuda":
            raise ValueError("token tensors must be CUDA tensors")
        if t.dtype != q.dtype:
            raise TypeError("all token tensors must share one dtype")
        if t.device != q.device:
            raise ValueError("all tensors must be on one device")


def _channel_contiguous(ts):
    return [t if t.stride(-1) == 1 or t.shape[-1] == 1 else t.contiguous() for t in ts]


def _same_strides(group):
    """The ABI shares one stride triple per group; make the group agree."""
    s0 = group[0].stride()[:3]
    if all(t.stride()[:3] == s0 for t in group):
        return group
    return [t.contiguous() for t in group]


def _dims(q, k, v, o, packed: _Packed) -> N.LaDims:
    """q (and dq) give qk_strides, o (and do) v_strides; with grouped key/value
    heads k (dk) and v (dv) have strides of their own."""
    B, T, H, D = q.shape
    E = v.shape[3]
    d = N.LaDims()
    d.batch, d.seq_len, d.heads, d.dim_qk, d.dim_v = B, T, H, D, E
    d.num_seqs = packed.n
    grouped = k.shape[2] != H
    d.kv_heads = k.shape[2] if grouped else 0
    for i in range(3):
        d.qk_strides[i] = q.stride(i)
        d.v_strides[i] = o.stride(i)
        if grouped:
            d.k_strides[i] = k.stride(i)
            d.kv_v_strides[i] = v.stride(i)
    return d


def _state(x: Optional[Tensor], shape, device, name) -> Optional[Tensor]:
    if x is None:
        return None
    if tuple(x.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(x.shape)))
    return x.to(device=device, dtype=torch.float32).contiguous()


def _g(g_gamma, H, device) -> Tensor:
    g = torch.as_tensor(g_gamma, dtype=torch.float32)
    if g.numel() == 1 and H != 1:
        g = g.reshape(1).expand(H)
    if tuple(g.shape) != (H,):
        raise ValueError("g_gamma must have shape [num_heads] = [%d]" % H)
    return g.to(device).contiguous()


def _num_states(q, packed):
    return packed.n if packed.dev is not None else q.shape[0]


def _like(t: Tensor) -> Tensor:
    """Uninitialised output with t's shape, dtype and (dense) strides."""
    return torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, device=t.device)


@_traced
def la_fwd(q: Tensor, k: Tensor, v: Tensor, g_gamma, scale: Optional[float] = None,
           initial_state: Optional[Tensor] = None, reverse: bool = False,
           cu_seqlens=None, out: Optional[Tensor] = None,
           final_state: Optional[Tensor] = None, want_final_state: bool = True,
           workspace: bool = True) -> Tuple[Tensor, Optional[Tensor]]:
    """Forward pass. q, k: [B,T,H,D]; v: [B,T,H,E]; returns (o [B,T,H,E], final [N,H,D,E]).
    workspace=False passes no device workspace: packed sequences then run in index
    order (no longest-first schedule) and never split."""
    _check_tokens(q, k, v)
    q, k, v = _channel_contiguous((q, k, v))
    grouped = k.shape[2] != q.shape[2]
    if not grouped:
        q, k = _same_strides([q, k])
    dev = q.device
    packed = _Packed(cu_seqlens, dev)
    B, T, H, D = q.shape
    E = v.shape[3]
    Nst = _num_states(q, packed)
    g = _g(g_gamma, H, dev)
    scale = float(D ** -0.5 if scale is None else scale)
    init = _state(initial_state, (Nst, H, D, E), dev, "initial_state")
    o_shape = q.shape[:3] + v.shape[3:]
    if out is None:
        out = _like(v) if not grouped else torch.empty(o_shape, dtype=v.dtype, device=dev)
    if (tuple(out.shape) != tuple(o_shape) or out.dtype != v.dtype or out.stride(-1) != 1
            or (not grouped and out.stride()[:3] != v.stride()[:3])):
        raise ValueError("out must be [B, T, H, E] of v's dtype (with v's strides when keys "
                         "and values have H heads)")
    if final_state is None and want_final_state:
        final_state = torch.empty((Nst, H, D, E), device=dev, dtype=torch.float32)
    dims = _dims(q, k, v, out, packed)
    ws = packed.ws_args(dims, _dtype_code(q)) if workspace else (None, 0)
    st = N.lib().la_fwd(ctypes.byref(dims), _dtype_code(q), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                        scale, _ptr(init), int(bool(reverse)), _ptr(packed.dev),
                        packed.host_ptr(), _ptr(out), _ptr(final_state), *ws,
                        _stream(dev))
    N.check(st)
    return out, final_state


def _bwd_prep(q, k, v, do, g_gamma, scale, initial_state, d_final_state, cu_seqlens):
    _check_tokens(q, k, v, (do,))
    if tuple(do.shape) != tuple(q.shape[:3] + v.shape[3:]):
        raise ValueError("do must be [B, T, H, E]")
    q, k, v, do = _channel_contiguous((q, k, v, do))
    if k.shape[2] == q.shape[2]:
        q, k = _same_strides([q, k])
        v, do = _same_strides([v, do])
    dev = q.device
    packed = _Packed(cu_seqlens, dev)
    B, T, H, D = q.shape
    E = v.shape[3]
    Nst = _num_states(q, packed)
    g = _g(g_gamma, H, dev)
    scale = float(D ** -0.5 if scale is None else scale)
    init = _state(initial_state, (Nst, H, D, E), dev, "initial_state")
    dfin = _state(d_final_state, (Nst, H, D, E), dev, "d_final_state")
    return q, k, v, do, dev, packed, g, scale, init, dfin, Nst


@_traced
def la_bwd(q: Tensor, k: Tensor, v: Tensor, do: Tensor, g_gamma, scale: Optional[float] = None,
           initial_state: Optional[Tensor] = None, d_final_state: Optional[Tensor] = None,
           reverse: bool = False, cu_seqlens=None, want_d_initial_state: bool = True,
           workspace: bool = True):
    """Backward pass: returns (dq, dk, dv, d_initial_state) of
    sum(o*do) + sum(final_state*d_final_state).  workspace=False as in la_fwd (not
    with grouped key/value heads, which need it)."""
    q, k, v, do, dev, packed, g, scale, init, dfin, Nst = _bwd_prep(
        q, k, v, do, g_gamma, scale, initial_state, d_final_state, cu_seqlens)
    dq, dk, dv = _like(q), _like(k), _like(v)
    dinit = (torch.empty((Nst, q.shape[2], q.shape[3], v.shape[3]), device=dev,
                         dtype=torch.float32) if want_d_initial_state else None)
    dims = _dims(q, k, v, do, packed)
    ws = packed.ws_args(dims, _dtype_code(q)) if workspace else (None, 0)
    st = N.lib().la_bwd(ctypes.byref(dims), _dtype_code(q), _ptr(q), _ptr(k), _ptr(v), _ptr(do),
                        _ptr(g), scale, _ptr(init), _ptr(dfin), int(bool(reverse)),
                        _ptr(packed.dev), packed.host_ptr(), _ptr(dq), _ptr(dk), _ptr(dv),
                        _ptr(dinit), *ws, _stream(dev))
    N.check(st)
    return dq, dk, dv, dinit


@_traced
def la_bwd_dq(q, k, v, do, g_gamma, scale=None, initial_state=None, reverse=False,
              cu_seqlens=None):
    """dq only (one sweep in processing order)."""
    q, k, v, do, dev, packed, g, scale, init, _, _ = _bwd_prep(
        q, k, v, do, g_gamma, scale, initial_state, None, cu_seqlens)
    dq = _like(q)
    dims = _dims(q, k, v, do, packed)
    ws = packed.ws_args(dims, _dtype_code(q))
    st = N.lib().la_bwd_dq(ctypes.byref(dims), _dtype_code(q), _ptr(q), _ptr(k), _ptr(v),
                           _ptr(do), _ptr(g), scale, _ptr(init), int(bool(reverse)),
                           _ptr(packed.dev), packed.host_ptr(), _ptr(dq), *ws,
                           _stream(dev))
    N.check(st)
    return dq


@_traced
def la_bwd_dkdv(q, k, v, do, g_gamma, scale=None, d_final_state=None, reverse=False,
                cu_seqlens=None, want_d_initial_state=True):
    """dk, dv and d_initial_state (one sweep against processing order)."""
    q, k, v, do, dev, packed, g, scale, _, dfin, Nst = _bwd_prep(
        q, k, v, do, g_gamma, scale, None, d_final_state, cu_seqlens)
    dk, dv = _like(k), _like(v)
    dinit = (torch.empty((Nst, q.shape[2], q.shape[3], v.shape[3]), device=dev,
                         dtype=torch.float32) if want_d_initial_state else None)
    dims = _dims(q, k, v, do, packed)
    ws = packed.ws_args(dims, _dtype_code(q))
    st = N.lib().la_bwd_dkdv(ctypes.byref(dims), _dtype_code(q), _ptr(q), _ptr(k), _ptr(v),
                             _ptr(do), _ptr(g), scale, _ptr(dfin), int(bool(reverse)),
                             _ptr(packed.dev), packed.host_ptr(), _ptr(dk), _ptr(dv),
                             _ptr(dinit), *ws, _stream(dev))
    N.check(st)
    return dk, dv, dinit


def get_device_error(device=None) -> None:
    """Raises LaError(LA_ERR_TIMEOUT) if an on-device bounded wait ran out."""
    N.check(N.lib().la_get_device_error(_stream(device)))


def kernel_family(B, T, H, D, E, dtype=torch.bfloat16, layout="bthd") -> int:
    """2 = token-by-token kernels (T <= 16), 1 = tensor-core chunked kernels,
    0 = CUDA-core chunked kernels, -1 = unsupported."""
    d = N.LaDims()
    d.batch, d.seq_len, d.heads, d.dim_qk, d.dim_v, d.num_seqs = B, T, H, D, E, 0
    if layout == "bthd":
        qs, vs = (T * H * D, H * D, D), (T * H * E, H * E, E)
    else:  # bhtd
        qs, vs = (H * T * D, D, T * D), (H * T * E, E, T * E)
    for i in range(3):
        d.qk_strides[i] = qs[i]
        d.v_strides[i] = vs[i]
    code = N.LA_DTYPE_BF16 if dtype == torch.bfloat16 else N.LA_DTYPE_F32
    return int(N.lib().la_kernel_family(ctypes.byref(d), code))


def _gate(g, q):
    """The per-key gate as fp32 with a contiguous channel dimension."""
    if tuple(g.shape) != tuple(q.shape):
        raise ValueError("g must have the queries' shape %s, got %s"
                         % (tuple(q.shape), tuple(g.shape)))
    g = g.to(device=q.device, dtype=torch.float32)
    return g if g.stride(-1) == 1 else g.contiguous()


def _strides3(t):
    return (ctypes.c_int64 * 3)(*t.stride()[:3])


@_traced
def gla_fwd(q: Tensor, k: Tensor, v: Tensor, g: Tensor, g_gamma=None,
            scale: Optional[float] = None, initial_state: Optional[Tensor] = None,
            reverse: bool = False, cu_seqlens=None, chunked: bool = True,
            keep_operands: bool = False):
    """Gated forward (GLA): row a of the state decays by exp(g_gamma[h] + g_t[a]) at
    token t.  q, g: [B,T,H,D]; k: [B,T,H_kv,D], v: [B,T,H_kv,E] with H_kv dividing H
    (query head h reads key/value head h // (H / H_kv); the gate and the state are
    the query head's).  Returns (o, final_state), and with
    keep_operands=True (o, final_state, operands): operands is the workspace holding
    the chunked form's rescaled q, k when the call ran that form (else None), to be
    passed once to gla_bwd on the same inputs.  chunked=False withholds the
    workspace, so that every (sequence, head) runs token by token (otherwise the
    chunked tensor-core form runs where it applies)."""
    _check_tokens(q, k, v)
    q, k, v = _channel_contiguous((q, k, v))
    if k.shape[2] == q.shape[2]:
        q, k = _same_strides([q, k])
    dev = q.device
    g = _gate(g, q)
    packed = _Packed(cu_seqlens, dev)
    B, T, H, D = q.shape
    E = v.shape[3]
    Nst = _num_states(q, packed)
    gg = _g(torch.zeros(H) if g_gamma is None else g_gamma, H, dev)
    scale = float(D ** -0.5 if scale is None else scale)
    init = _state(initial_state, (Nst, H, D, E), dev, "initial_state")
    # o has the queries' heads; with H heads for keys and values too, v's strides
    out = (_like(v) if k.shape[2] == H
           else torch.empty(q.shape[:3] + v.shape[3:], dtype=v.dtype, device=dev))
    fin = torch.empty((Nst, H, D, E), device=dev, dtype=torch.float32)
    dims = _dims(q, k, v, out, packed)
    gs = _strides3(g)
    nbytes = (int(N.lib().la_gla_fwd_workspace_size(ctypes.byref(dims), _dtype_code(q),
                                                    packed.host_ptr())) if chunked else 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
    written = ctypes.c_int32(0)
    st = N.lib().la_gla_fwd(ctypes.byref(dims), _dtype_code(q), _ptr(q), _ptr(k), _ptr(v),
                            _ptr(g), gs, _ptr(gg), scale, _ptr(init), int(bool(reverse)),
                            _ptr(packed.dev), packed.host_ptr(), _ptr(out), _ptr(fin),
                            _ptr(ws), nbytes, ctypes.byref(written), _stream(dev))
    N.check(st)
    if keep_operands:
        return out, fin, (ws if written.value else None)
    return out, fin


@_traced
def gla_bwd(q, k, v, do, g, g_gamma=None, scale=None, initial_state=None, d_final_state=None,
            reverse=False, cu_seqlens=None, want_d_initial_state=True, operands=None,
            chunked: bool = True):
    """Backward of gla_fwd: returns (dq, dk, dv, dg, d_initial_state); with grouped
    key/value heads dk and dv are the sums over each group's query heads.  operands: what
    gla_fwd(..., keep_operands=True) returned for the same inputs, or None; it is
    consumed (used as scratch).  chunked=False (with operands None) gives only the
    token-by-token part of the workspace, so that every (sequence, head) runs token
    by token."""
    if not chunked and operands is not None:
        raise ValueError("chunked=False takes no operands")
    q, k, v, do, dev, packed, gg, scale, init, dfin, Nst = _bwd_prep(
        q, k, v, do, torch.zeros(q.shape[2]) if g_gamma is None else g_gamma, scale,
        initial_state, d_final_state, cu_seqlens)
    g = _gate(g, q)
    dq, dk, dv = _like(q), _like(k), _like(v)
    dg = torch.empty_strided(g.shape, g.stride(), dtype=torch.float32, device=dev)
    dinit = (torch.empty((Nst, q.shape[2], q.shape[3], v.shape[3]), device=dev,
                         dtype=torch.float32) if want_d_initial_state else None)
    dims = _dims(q, k, v, do, packed)
    # with the forward's operands the workspace needs only the token-by-token part
    nbytes = int(N.lib().la_gla_workspace_size(ctypes.byref(dims), _dtype_code(q),
                                              packed.host_ptr(),
                                              int(operands is not None or not chunked)))
    fwd_bytes = operands.numel() if operands is not None else 0
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    st = N.lib().la_gla_bwd(ctypes.byref(dims), _dtype_code(q), _ptr(q), _ptr(k), _ptr(v),
                            _ptr(do), _ptr(g), _strides3(g), _ptr(gg), scale, _ptr(init),
                            _ptr(dfin), int(bool(reverse)), _ptr(packed.dev), packed.host_ptr(),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dinit),
                            ctypes.c_void_p(ws.data_ptr()), nbytes, _ptr(operands), fwd_bytes,
                            _stream(dev))
    N.check(st)
    return dq, dk, dv, dg, dinit


class _GatedLinearAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, init, gg, scale, reverse, cu):
        o, fin, ops = gla_fwd(q, k, v, g, gg, scale, init, reverse, cu, keep_operands=True)
        ctx.save_for_backward(q, k, v, g, init, gg)
        ctx.scale, ctx.reverse, ctx.cu = scale, reverse, cu
        ctx.has_init = init is not None
        ctx.ops = ops   # the chunked form's operands, reused once by the backward
        return o, fin

    @staticmethod
    def backward(ctx, do, dfin):
        q, k, v, g, init, gg = ctx.saved_tensors
        if do is None:
            do = torch.zeros(q.shape[:3] + v.shape[3:], dtype=v.dtype, device=v.device)
        ops, ctx.ops = ctx.ops, None
        dq, dk, dv, dg, dinit = gla_bwd(q, k, v, do.to(v.dtype), g, gg, ctx.scale,
                                        init if ctx.has_init else None, dfin, ctx.reverse,
                                        ctx.cu, want_d_initial_state=ctx.has_init,
                                        operands=ops)
        return (dq, dk, dv, dg.to(g.dtype), (dinit if ctx.has_init else None), None, None,
                None, None)


class _LinearAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, init, g, scale, reverse, cu):
        o, fin = la_fwd(q, k, v, g, scale, init, reverse, cu)
        ctx.save_for_backward(q, k, v, init, g)
        ctx.scale, ctx.reverse, ctx.cu = scale, reverse, cu
        ctx.has_init = init is not None
        return o, fin

    @staticmethod
    def backward(ctx, do, dfin):
        q, k, v, init, g = ctx.saved_tensors
        if do is None:
            do = torch.zeros(q.shape[:3] + v.shape[3:], dtype=v.dtype, device=v.device)
        dq, dk, dv, dinit = la_bwd(q, k, v, do.to(v.dtype), g, ctx.scale,
                                   init if ctx.has_init else None, dfin, ctx.reverse, ctx.cu,
                                   want_d_initial_state=ctx.has_init)
        return dq, dk, dv, (dinit if ctx.has_init else None), None, None, None, None


def _packed_batch_msg(batch):
    return ("with cu_seqlens every sequence is packed into one batch row, so the batch "
            "dimension must be 1 (got %d)" % batch)


def _check_packing(query, cu_seqlens, initial_state):
    """A packed call (cu_seqlens given) holds every sequence in one batch row and,
    with an initial state, one state per sequence."""
    if cu_seqlens is None:
        return
    if query.ndim == 4 and query.shape[0] != 1:
        raise ValueError(_packed_batch_msg(query.shape[0]))
    n_seqs = len(cu_seqlens) - 1
    if initial_state is not None and initial_state.shape[0] != n_seqs:
        raise ValueError("initial_state needs one state per packed sequence: %d sequences, "
                         "%d states" % (n_seqs, initial_state.shape[0]))


def _scale_for(softmax_scale, head_dim):
    """The query scale: the caller's, else 1/sqrt(head width)."""
    return 1.0 / math.sqrt(head_dim) if softmax_scale is None else softmax_scale


def recurrent(query: Tensor, key: Tensor, value: Tensor, g=None, g_gamma=None, gk=None, gv=None,
              softmax_scale: Optional[float] = None, initial_state: Optional[Tensor] = None,
              reverse: bool = False, cu_seqlens=None):
    """ejkernel `recurrent` with the per-head `g_gamma` decay and the GLA-style gate `g`
    (a log-decay per key channel, [B,T,H,D]; gk / gv are not implemented).  Accepts
    [B,T,H,D] or packed [T_total,H,D] with cu_seqlens.  Returns (o, final_state);
    differentiable in query, key, value, g and initial_state."""
    if gk is not None or gv is not None:
        raise NotImplementedError("the gk / gv gates are not implemented")
    squeeze = False
    if query.ndim == 3:
        if cu_seqlens is None:
            raise ValueError("3-D inputs need cu_seqlens")
        query, key, value = query[None], key[None], value[None]
        g = None if g is None else g[None]
        squeeze = True
    if cu_seqlens is not None and query.shape[0] != 1:
        raise ValueError(_packed_batch_msg(query.shape[0]))
    H = query.shape[2]
    if g_gamma is None:
        g_gamma = torch.zeros(H, dtype=torch.float32)
    gg = _g(g_gamma, H, query.device)
    softmax_scale = _scale_for(softmax_scale, query.shape[-1])
    if g is not None:
        o, fin = _GatedLinearAttention.apply(query, key, value, g, initial_state, gg,
                                             softmax_scale, bool(reverse), cu_seqlens)
    else:
        o, fin = _LinearAttention.apply(query, key, value, initial_state, gg, softmax_scale,
                                        bool(reverse), cu_seqlens)
    return (o[0] if squeeze else o), fin


def recurrent_gla(query: Tensor, key: Tensor, value: Tensor, g: Optional[Tensor] = None,
                  g_gamma=None, softmax_scale: Optional[float] = None,
                  initial_state: Optional[Tensor] = None, reverse: bool = False,
                  cu_seqlens=None):
    """ejkernel `recurrent_gla` (the GLA page): the batch-1 / initial-state count
    checks of that page, the default scale from the key width, then `recurrent`."""
    _check_packing(query, cu_seqlens, initial_state)
    return recurrent(query, key, value, g=g, g_gamma=g_gamma,
                     softmax_scale=_scale_for(softmax_scale, key.shape[-1]),
                     initial_state=initial_state, reverse=reverse, cu_seqlens=cu_seqlens)


def lightning_attn(query: Tensor, key: Tensor, value: Tensor, layer_idx: int, num_layers: int,
                   softmax_scale: Optional[float] = None, initial_state: Optional[Tensor] = None,
                   reverse: bool = False, cu_seqlens=None):
    """ejkernel `lightning_attn`: g_gamma from the layer position, then `recurrent`.
    Keys and values have the queries' shape (that page's docstring); grouped
    key/value heads go through `recurrent` or la_fwd / la_bwd."""
    if key.shape != query.shape or value.shape[:-1] != query.shape[:-1]:
        raise ValueError("lightning_attn: key must have the shape of query and value its "
                         "leading dims (got %s, %s, %s)"
                         % (tuple(query.shape), tuple(key.shape), tuple(value.shape)))
    _check_packing(query, cu_seqlens, initial_state)
    H = query.shape[-2]
    return recurrent(query, key, value, g_gamma=lightning_g_gamma(H, layer_idx, num_layers),
                     softmax_scale=_scale_for(softmax_scale, key.shape[-1]),
                     initial_state=initial_state, reverse=reverse, cu_seqlens=cu_seqlens)


def lightning_attn_func(q: Tensor, k: Tensor, v: Tensor, s: Tensor) -> Tensor:
    """Lightning-Attention-2 README call: q, k [b,h,n,d], v [b,h,n,e], slopes s [h]
    (decay exp(-s)), scale 1.  Returns o [b,h,n,e]; differentiable."""
    g = -torch.as_tensor(s, dtype=torch.float32).reshape(-1)
    # (b, h, n, d) -> (b, n, h, d) views: no copy, the ABI takes the strides.
    o, _ = _LinearAttention.apply(q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), None,
                                  g.to(q.device), 1.0, False, None)
    return o.transpose(1, 2)
