"""The drop-in for torch.nn.functional.scaled_dot_product_attention: argument
handling on the host (no GPU), and a small attention layer run through the
patched function on the GPU: its attention output and the gradients of the
attention's inputs compared element by element with the fp64 oracle on the
exact bf16 values the layer handed to attention."""
import math

import numpy as np
import pytest
import torch

import oracle
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
    384 tokens x 64 per head, bf16.  What the patched attention received (q, k,
    v as strided views of the projections) and returned (o), and the gradients
    autograd sent into it (dO) and out of it (dq, dk, dv), are captured; o and
    dq, dk, dv must match the oracle on those inputs within 2e-2."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(11)
    B, H, N, d = 2, 4, 384, 64
    x = torch.randn(B, N, H * d, device=dev, generator=g, dtype=torch.float32)
    w = [torch.randn(H * d, H * d, device=dev, generator=g) / math.sqrt(H * d) for _ in range(4)]
    seen = {}

    def layer(inp):
        xb = inp.to(torch.bfloat16)
        q, k, v = ((xb @ wi.to(torch.bfloat16).T).view(B, N, H, d).transpose(1, 2) for wi in w[:3])
        for name, z in (("q", q), ("k", k), ("v", v)):
            z.retain_grad()
            seen[name] = z
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)
        seen["o"] = o
        o.register_hook(lambda grad: seen.__setitem__("dO", grad.detach().clone()))
        return (o.transpose(1, 2).reshape(B, N, H * d) @ w[3].to(torch.bfloat16).T).float()

    x1 = x.clone().requires_grad_(True)
    with fa_autograd.patch_sdpa():
        y1 = layer(x1)
        y1.square().mean().backward()
    torch.cuda.synchronize()
    f64 = lambda z: z.detach().double().cpu().numpy().reshape(B * H, N, d)   # noqa: E731
    Q, K, V, dO = f64(seen["q"]), f64(seen["k"]), f64(seen["v"]), f64(seen["dO"])
    dQ, dK, dV, O, L, _ = oracle.attn_bwd_ref(Q, K, V, dO, 1.0 / math.sqrt(d), causal)
    for name, got, want in (("O", seen["o"], O), ("dQ", seen["q"].grad, dQ), ("dK", seen["k"].grad, dK),
                            ("dV", seen["v"].grad, dV)):
        gv = f64(got)
        bad = np.abs(gv - want) > 2e-2 + 2e-2 * np.abs(want)
        assert not bad.any(), f"{name}: {bad.sum()} of {bad.size} outside 2e-2 (max {np.abs(gv - want).max():.3g})"
