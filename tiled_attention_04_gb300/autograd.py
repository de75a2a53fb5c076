"""FlashAttention as a torch.autograd.Function over the C ABI.

Interface of CS336 A2 "Systems and Parallelism", problem flash_forward:
``forward(ctx, Q, K, V, is_causal=False)`` returns O, saves L with
``ctx.save_for_backward`` (the only saved tensor of shape (batch, n_queries))
and stashes ``ctx.is_causal``; ``backward`` returns dQ, dK, dV (problem
flash_backward).  Inputs are (..., N, d) CUDA tensors, fp32 or bf16.
"""
from __future__ import annotations

import torch

from . import binding


class FlashAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Q, K, V, is_causal=False):
        Q, K, V = Q.contiguous(), K.contiguous(), V.contiguous()
        O, L = binding.fa_fwd(Q, K, V, is_causal=is_causal)
        ctx.save_for_backward(Q, K, V, O, L)
        ctx.is_causal = bool(is_causal)
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, O, L = ctx.saved_tensors
        dQ, dK, dV = binding.fa_bwd(Q, K, V, O, dO.contiguous(), L, is_causal=ctx.is_causal)
        return dQ, dK, dV, None


def flash_attention(Q, K, V, is_causal=False):
    return FlashAttention.apply(Q, K, V, is_causal)
