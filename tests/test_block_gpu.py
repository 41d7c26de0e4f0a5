"""The attention layer (QKV projection -> Fibottention -> output projection)
against the same layer with the attention core written as masked dense
softmax attention in torch (mask from the oracle's support), same weights:
outputs and every gradient (input and parameters)."""
import numpy as np
import pytest
import torch

import oracle
from sparse_head_self_gb300.block import FibottentionSelfAttention

pytestmark = pytest.mark.gpu


def _dense_layer_reference(layer, x, heads_list, global_token):
    B, N, dim = x.shape
    H = layer.heads
    qkv = layer.qkv(x).view(B, N, 3, H, 64).permute(2, 0, 3, 1, 4)
    q, k, v = qkv[0], qkv[1], qkv[2]
    masks = torch.stack([torch.from_numpy(oracle.support_mask(N, h).astype(bool)) for h in heads_list]).to(x.device)
    s = (layer.scale * q @ k.transpose(-1, -2)).masked_fill(~masks[None], float("-inf"))
    p = torch.softmax(s, dim=-1).nan_to_num(0.0)
    o = p @ v
    return layer.proj(o.transpose(1, 2).reshape(B, N, dim))


@pytest.mark.parametrize("global_token", [False, True])
def test_layer_matches_dense_masked_reference(global_token):
    torch.manual_seed(0)
    B, H, N = 3, 4, 197
    layer = FibottentionSelfAttention(H * 64, H, N, 5, 197, True, global_token=global_token).cuda()
    w = oracle.windows(H, 5, 197)
    heads = [oracle.Head.fibottention(*oracle.wythoff_row(i + 1), w[i], True, global_token) for i in range(H)]
    x = torch.randn(B, N, H * 64, device="cuda", requires_grad=True)
    y = layer(x)
    g = torch.randn_like(y)
    y.backward(g)
    grads = [x.grad.clone()] + [p.grad.clone() for p in layer.parameters()]
    x.grad = None
    layer.zero_grad()
    y_ref = _dense_layer_reference(layer, x, heads, global_token)
    y_ref.backward(g)
    grads_ref = [x.grad] + [p.grad for p in layer.parameters()]
    torch.testing.assert_close(y, y_ref, atol=2e-4, rtol=1e-4)
    for a, b in zip(grads, grads_ref):
        torch.testing.assert_close(a, b, atol=2e-3, rtol=1e-3)


def test_layer_bf16_runs_and_is_close():
    torch.manual_seed(1)
    B, H, N = 2, 12, 197
    layer = FibottentionSelfAttention(H * 64, H, N, 5, 197, True).cuda()
    x = torch.randn(B, N, H * 64, device="cuda")
    y32 = layer(x)
    y16 = layer.to(torch.bfloat16)(x.to(torch.bfloat16))
    assert y16.dtype == torch.bfloat16
    d = (y16.float() - y32).abs()
    assert float(d.mean()) < 2e-2
