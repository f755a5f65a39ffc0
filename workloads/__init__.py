"""Seeded synthetic inputs for decayed causal linear attention.

This module is the only code that both the CUDA path (tests, bench) and the
CPU oracle consume.  It draws random tensors and writes down the workload
recipes (shapes, decay slopes, scales); it holds none of the method's
arithmetic.  Every tensor is drawn on the CPU from torch.Generator seeded
with `seed`, in the order q, k, v, do, initial_state, d_final_state, and
then cast to the workload's dtype, so that the oracle (which upcasts the
cast values to fp64) and the GPU (which receives the cast values) see
identical numbers.

Decay recipes, as the pages give them:
  * Lightning layer-dependent decay (ejkernel lightning_attn, module
    docstring, the decay formula):
        g_gamma[h] = -(8 / H) * (1 - layer_idx / num_layers) * h
  * ALiBi-style slopes (Lightning-Attention README, usage section:
    `_build_slope_tensor(h)`, decay = exp(-slope)); the slope list itself is
    not printed, the workload uses s_i = 2^(-8 i / H), i = 1..H.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


def lightning_g_gamma(H: int, layer_idx: int, num_layers: int) -> torch.Tensor:
    return -(8.0 / H * (1.0 - layer_idx / num_layers)) * torch.arange(H, dtype=torch.float32)


def alibi_g_gamma(H: int) -> torch.Tensor:
    i = torch.arange(1, H + 1, dtype=torch.float64)
    return (-(2.0 ** (-8.0 * i / H))).to(torch.float32)


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    T: int
    H: int
    d: int
    e: int
    dtype: torch.dtype
    g_gamma: torch.Tensor
    scale: float
    seqlens: Optional[list] = None        # packed varlen lengths (B = 1)
    init_std: float = 0.0                 # 0: no initial_state
    dfinal_std: float = 0.0               # 0: no d_final_state
    backward: bool = True

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens) if self.seqlens is not None else self.B

    @property
    def cu_seqlens(self) -> Optional[torch.Tensor]:
        if self.seqlens is None:
            return None
        cu = [0]
        for L in self.seqlens:
            cu.append(cu[-1] + int(L))
        return torch.tensor(cu, dtype=torch.int32)

    @property
    def tokens(self) -> int:
        return self.B * self.T


def tiny_fp32() -> Workload:
    """b=1 h=2 n=256 d=e=32 fp32, Lightning decay (layer 5 of 12), forward only."""
    return Workload("tiny_fp32_b1_h2_n256_d32", 1, 256, 2, 32, 32, torch.float32,
                    lightning_g_gamma(2, 5, 12), 1.0 / math.sqrt(32), backward=False)


def small_bf16() -> Workload:
    """b=2 h=8 n=2048 d=e=64 bf16, Lightning decay (layer 5 of 12), fwd+bwd."""
    return Workload("b2_h8_n2048_d64_bf16", 2, 2048, 8, 64, 64, torch.bfloat16,
                    lightning_g_gamma(8, 5, 12), 1.0 / 8.0)


def sweep_bf16(n: int) -> Workload:
    """b=4 h=32 d=e=128 bf16, ALiBi slopes, scale 1: the Lightning-2 benchmark shape."""
    return Workload("b4_h32_n%d_d128_bf16" % n, 4, n, 32, 128, 128, torch.bfloat16,
                    alibi_g_gamma(32), 1.0)


SWEEP_LENGTHS = (512, 1024, 2048, 4096, 8192, 16384, 32768)


def d192_bf16() -> Workload:
    """b=2 h=12 n=2048 d=e=192 bf16 (the README usage example's shape), ALiBi slopes."""
    return Workload("b2_h12_n2048_d192_bf16", 2, 2048, 12, 192, 192, torch.bfloat16,
                    alibi_g_gamma(12), 1.0 / math.sqrt(192))


def varlen_bf16(seed: int = 0, num_seqs: int = 16, lo: int = 64, hi: int = 8192) -> Workload:
    """16 packed sequences, lengths uniform in [64, 8192] from the seed, h=16 d=e=128
    bf16, initial_state ~ N(0, 0.02^2), Lightning decay (layer 3 of 24)."""
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(lo, hi + 1, (num_seqs,), generator=gen).tolist()
    return Workload("varlen16_h16_d128_bf16", 1, int(sum(lens)), 16, 128, 128, torch.bfloat16,
                    lightning_g_gamma(16, 3, 24), 1.0 / math.sqrt(128), seqlens=lens,
                    init_std=0.02, dfinal_std=0.02)


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu") -> dict:
    """Draw q, k, v, do (N(0,1)), initial_state and d_final_state (fp32, N(0, std^2)
    when the workload asks for them) in that order; cast to w.dtype."""
    gen = torch.Generator().manual_seed(seed)
    shp_qk = (w.B, w.T, w.H, w.d)
    shp_v = (w.B, w.T, w.H, w.e)
    q = torch.randn(shp_qk, generator=gen).to(w.dtype)
    k = torch.randn(shp_qk, generator=gen).to(w.dtype)
    v = torch.randn(shp_v, generator=gen).to(w.dtype)
    do = torch.randn(shp_v, generator=gen).to(w.dtype) if w.backward else None
    shp_s = (w.num_seqs, w.H, w.d, w.e)
    init = torch.randn(shp_s, generator=gen) * w.init_std if w.init_std > 0 else None
    dfin = (torch.randn(shp_s, generator=gen) * w.dfinal_std
            if (w.dfinal_std > 0 and w.backward) else None)
    out = dict(q=q, k=k, v=v, do=do, initial_state=init, d_final_state=dfin,
               g_gamma=w.g_gamma.clone(), scale=w.scale, cu_seqlens=w.cu_seqlens)
    if device != "cpu":
        out = {n: (t.to(device) if isinstance(t, torch.Tensor) else t) for n, t in out.items()}
        if w.cu_seqlens is not None:
            out["cu_seqlens_host"] = w.cu_seqlens
    return out


def random_small(seed: int, B: int, T: int, H: int, d: int, e: int,
                 dtype=torch.float64, g_lo: float = -1.0, g_hi: float = 0.0) -> dict:
    """Tiny random problem for oracle pins: g_gamma uniform in [g_lo, g_hi]."""
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn((B, T, H, d), generator=gen, dtype=torch.float64).to(dtype)
    k = torch.randn((B, T, H, d), generator=gen, dtype=torch.float64).to(dtype)
    v = torch.randn((B, T, H, e), generator=gen, dtype=torch.float64).to(dtype)
    do = torch.randn((B, T, H, e), generator=gen, dtype=torch.float64).to(dtype)
    g = g_lo + (g_hi - g_lo) * torch.rand((H,), generator=gen, dtype=torch.float64)
    return dict(q=q, k=k, v=v, do=do, g_gamma=g)
