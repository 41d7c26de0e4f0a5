"""A drop-in multi-head self-attention layer whose attention core is
Fibottention (the paper's Sec. 3 applied in a ViT encoder block: the QKV
projection, per-head attention over the Fibonacci support, the output
projection W^Z; README Algorithm 3 shows the same sequence of steps).

The projections are ordinary torch GEMMs; the attention core calls libfibatt
through ``fibottention`` (forward fibatt_fwd, backward fibatt_bwd).  Head i of
the layer uses Wythoff row pi(i) with the linear window schedule (paper
Sec. 3: a per-layer permutation pi of the heads is allowed).
"""
from __future__ import annotations

import torch
from torch import nn

from .api import HEAD_DIM, Support, fibottention


class FibottentionSelfAttention(nn.Module):
    """x [B, N, dim] -> [B, N, dim] with dim = heads * 64."""

    def __init__(self, dim: int, heads: int, N: int, w_min: int, w_max: int, include_diag: bool = True,
                 global_token: bool = False, modified: bool = False, permutation=None, bias: bool = True):
        super().__init__()
        if dim != heads * HEAD_DIM:
            raise ValueError(f"dim must be heads * {HEAD_DIM}")
        self.heads, self.N = heads, N
        self.qkv = nn.Linear(dim, 3 * dim, bias=bias)
        self.proj = nn.Linear(dim, dim, bias=bias)
        self.support = Support.wythoff(heads, N, w_min, w_max, include_diag, modified=modified,
                                       permutation=permutation).set_global_token(global_token)
        self.scale = HEAD_DIM ** -0.5

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        B, N, dim = x.shape
        if N != self.N:
            raise ValueError(f"sequence length {N}, layer built for {self.N}")
        qkv = self.qkv(x).view(B, N, 3, self.heads, HEAD_DIM).permute(2, 0, 3, 1, 4)
        q, k, v = (t.contiguous() for t in qkv)            # [B, H, N, 64] each
        o = fibottention(q, k, v, self.support, self.scale)  # [B, H, N, 64]
        return self.proj(o.transpose(1, 2).reshape(B, N, dim))


__all__ = ["FibottentionSelfAttention"]
