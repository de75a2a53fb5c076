"""FlashAttention as a torch.autograd.Function over the C ABI.

Interface of CS336 A2 "Systems and Parallelism", problem flash_forward:
``forward(ctx, Q, K, V, is_causal=False)`` returns O, saves L with
``ctx.save_for_backward`` (the only saved tensor of shape (batch, n_queries))
and stashes ``ctx.is_causal``; ``backward`` returns dQ, dK, dV (problem
flash_backward).  Inputs are (..., N, d) CUDA tensors, fp32 or bf16; strided
(B, H, N, d) views (a projection's (B, N, H, d) output transposed, or slices
of a fused QKV projection) are read in place, without a reshape copy.

``scaled_dot_product_attention`` and ``patch_sdpa`` make it a drop-in for the
module-level attention function a Transformer layer calls (the field guide's
"Systems and Parallelism" §1.3 asks for the attention in the model to be
swapped for the flash kernel).
"""
from __future__ import annotations

import contextlib

import torch

from . import binding


def _in_place(t):
    """t itself when the kernels can read it where it lies (contiguous, or a strided
    (B, H, N, d) view such as a transposed projection output), else a fresh
    contiguous copy (a fresh allocation, so also 16-byte aligned)."""
    return t if binding.accepts_view(t) else t.clone(memory_format=torch.contiguous_format)


class FlashAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Q, K, V, is_causal=False, scale=None):
        Q, K, V = _in_place(Q), _in_place(K), _in_place(V)
        O, L = binding.fa_fwd(Q, K, V, is_causal=is_causal, scale=scale)
        ctx.save_for_backward(Q, K, V, O, L)
        ctx.is_causal = bool(is_causal)
        ctx.scale = scale
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, O, L = ctx.saved_tensors
        dQ, dK, dV = binding.fa_bwd(Q, K, V, O, _in_place(dO), L, is_causal=ctx.is_causal, scale=ctx.scale)
        return dQ, dK, dV, None, None


def flash_attention(Q, K, V, is_causal=False, scale=None):
    return FlashAttention.apply(Q, K, V, is_causal, scale)


def scaled_dot_product_attention(query, key, value, attn_mask=None, dropout_p=0.0, is_causal=False, scale=None,
                                 enable_gqa=False):
    """The arguments of torch.nn.functional.scaled_dot_product_attention that the
    method covers: no explicit mask (``is_causal`` gives the top-left causal one),
    no dropout, the same number of heads in query and key/value, and equal
    batch and head sizes.  Anything else raises ValueError."""
    if attn_mask is not None:
        raise ValueError("flash attention: an explicit attn_mask is not supported (use is_causal)")
    if dropout_p != 0.0:
        raise ValueError("flash attention: dropout is not supported")
    if enable_gqa or query.shape[:-2] != key.shape[:-2] or key.shape[:-2] != value.shape[:-2]:
        raise ValueError("flash attention: query, key and value need the same batch and head sizes")
    if key.shape[-1] != query.shape[-1] or value.shape[-1] != query.shape[-1]:
        raise ValueError("flash attention: query, key and value need the same head dimension")
    return FlashAttention.apply(query, key, value, is_causal, scale)


@contextlib.contextmanager
def patch_sdpa(fallback: bool = False):
    """Within the block, torch.nn.functional.scaled_dot_product_attention runs
    these kernels.  With ``fallback`` true, calls with arguments the method does
    not cover go to the original function instead of raising."""
    original = torch.nn.functional.scaled_dot_product_attention

    def patched(query, key, value, attn_mask=None, dropout_p=0.0, is_causal=False, scale=None, enable_gqa=False):
        try:
            return scaled_dot_product_attention(query, key, value, attn_mask, dropout_p, is_causal, scale,
                                                enable_gqa)
        except ValueError:
            if not fallback:
                raise
            return original(query, key, value, attn_mask=attn_mask, dropout_p=dropout_p, is_causal=is_causal,
                            scale=scale, enable_gqa=enable_gqa)

    torch.nn.functional.scaled_dot_product_attention = patched
    try:
        yield patched
    finally:
        torch.nn.functional.scaled_dot_product_attention = original
