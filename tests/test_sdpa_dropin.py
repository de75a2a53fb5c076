"""The drop-in for torch.nn.functional.scaled_dot_product_attention: argument
handling on the host (no GPU), and a small attention layer run through the
patched function on the GPU against torch's own attention."""
import math

import pytest
import torch

from tiled_attention_04_gb300 import autograd as fa_autograd


def test_patch_swaps_and_restores_the_module_function():
    original = torch.nn.functional.scaled_dot_product_attention
    with fa_autograd.patch_sdpa() as patched:
        assert torch.nn.functional.scaled_dot_product_attention is patched
    assert torch.nn.functional.scaled_dot_product_attention is original


@pytest.mark.parametrize("kwargs", [{"attn_mask": torch.zeros(4, 4)}, {"dropout_p": 0.1}, {"enable_gqa": True}])
def test_arguments_outside_the_method_are_refused_before_any_launch(kwargs):
    q = torch.zeros(1, 2, 4, 16)
    with pytest.raises(ValueError):
        fa_autograd.scaled_dot_product_attention(q, q, q, **kwargs)


def test_mismatched_heads_are_refused():
    q, k = torch.zeros(1, 4, 8, 16), torch.zeros(1, 2, 8, 16)
    with pytest.raises(ValueError):
        fa_autograd.scaled_dot_product_attention(q, k, k)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [True, False])
def test_attention_layer_through_the_patched_function(cuda_lib, causal):
    """x -> q, k, v projections -> attention -> output projection, 2 x 4 heads x
    384 tokens x 64 per head, bf16; outputs and the gradient of x against the
    same layer with torch's attention."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(11)
    B, H, N, d = 2, 4, 384, 64
    x = torch.randn(B, N, H * d, device=dev, generator=g, dtype=torch.float32)
    w = [torch.randn(H * d, H * d, device=dev, generator=g) / math.sqrt(H * d) for _ in range(4)]

    def layer(inp):
        xb = inp.to(torch.bfloat16)
        q, k, v = ((xb @ wi.to(torch.bfloat16).T).view(B, N, H, d).transpose(1, 2) for wi in w[:3])
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)
        return (o.transpose(1, 2).reshape(B, N, H * d) @ w[3].to(torch.bfloat16).T).float()

    x1 = x.clone().requires_grad_(True)
    with fa_autograd.patch_sdpa():
        y1 = layer(x1)
        y1.square().mean().backward()
    x2 = x.clone().requires_grad_(True)
    y2 = layer(x2)
    y2.square().mean().backward()
    torch.cuda.synchronize()
    assert torch.allclose(y1, y2, rtol=2e-2, atol=2e-2), (y1 - y2).abs().max()
    gscale = x2.grad.abs().max()
    assert torch.allclose(x1.grad, x2.grad, rtol=5e-2, atol=2e-2 * gscale), (x1.grad - x2.grad).abs().max()
