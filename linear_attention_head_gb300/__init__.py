"""GB300-native causal linear attention with per-head scalar exponential decay.

S_t = exp(g_gamma[h]) * S_{t-1} + k_t^T v_t,  o_t = (scale * q_t) S_t, in the
chunked Lightning-2 form, forward and backward, as hand-written sm_103a CUDA
kernels behind a C ABI (include/la.h).  PyTorch supplies device memory and
streams only.
"""
from ._native import (LaDims, LaError, LaInvalidArgument, LaUnsupported, LA_DTYPE_BF16,
                      LA_DTYPE_F32, lib)
from .api import (alibi_g_gamma, get_device_error, gla_bwd, gla_fwd, kernel_family, la_bwd,
                  la_bwd_dkdv, la_bwd_dq, la_fwd, lightning_attn, lightning_attn_func,
                  lightning_g_gamma, recurrent, recurrent_gla)

__all__ = [
    "LaDims", "LaError", "LaInvalidArgument", "LaUnsupported", "LA_DTYPE_BF16", "LA_DTYPE_F32",
    "lib", "alibi_g_gamma", "get_device_error", "gla_bwd", "gla_fwd", "kernel_family", "la_bwd",
    "la_bwd_dkdv", "la_bwd_dq", "la_fwd", "lightning_attn", "lightning_attn_func",
    "lightning_g_gamma", "recurrent", "recurrent_gla",
]
