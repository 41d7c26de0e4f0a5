"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only names workload shapes and
draws the random tensors that both the CUDA path and the CPU oracle consume.

Recipe (the same for every workload): Q, K, V and dO are i.i.d. N(0, 1),
drawn in fp32 on the CPU by ``torch.Generator().manual_seed(s)`` with
s = seed for Q, seed+1 for K, seed+2 for V and seed+3 for dO, then rounded
to nearest-even into the workload's I/O dtype.  Heads use Wythoff rows
1..H and the linear window schedule between ``w_min`` and ``w_max``; token
counts follow the shapes on the pages (8x8 patches + CLS = 65, ViT-B 14x14 +
CLS = 197, 8 frames x 196 patches + CLS = 1569, 128x128 + CLS = 16385).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str          # "f32" or "bf16"
    w_min: int
    w_max: int
    diag: bool
    backward: bool      # whether the workload's step includes the backward pass
    scale: float = 0.125  # 1/sqrt(64)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_batch(self, B: int) -> "Workload":
        return replace(self, B=B)


WORKLOADS: dict[str, Workload] = {
    # 8x8 patches + CLS, fp32, heads on Wythoff rows 1..3, w = 5, 35, 65
    "tiny": Workload("tiny", 1, 3, 65, 64, "f32", 5, 65, True, True),
    # ViT-B shape, 14x14 patches + CLS
    "vitb": Workload("vitb", 64, 12, 197, 64, "bf16", 5, 197, True, True),
    "vitb_nodiag": Workload("vitb_nodiag", 64, 12, 197, 64, "bf16", 5, 197, False, True),
    # TimeSformer-like video shape, 8 frames x 196 patches + CLS
    "video": Workload("video", 8, 12, 1569, 64, "bf16", 16, 1569, True, True),
    # ViT-B training batch
    "train": Workload("train", 256, 12, 197, 64, "bf16", 5, 197, True, True),
    # 128x128 patches + CLS
    "long": Workload("long", 2, 16, 16385, 64, "bf16", 64, 16385, True, True),
}


def randn(shape, seed: int, dtype: torch.dtype) -> torch.Tensor:
    """N(0,1) in fp32 from a CPU generator seeded with ``seed``, then cast (RNE)."""
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    return x.to(dtype)


def make_inputs(wl: Workload, seed: int = 0, with_grad: bool = True):
    """CPU tensors (Q, K, V, dO) of shape [B, H, N, D] in the workload's dtype."""
    shape = (wl.B, wl.H, wl.N, wl.D)
    dt = wl.torch_dtype
    q = randn(shape, seed, dt)
    k = randn(shape, seed + 1, dt)
    v = randn(shape, seed + 2, dt)
    do = randn(shape, seed + 3, dt) if with_grad else None
    return q, k, v, do
