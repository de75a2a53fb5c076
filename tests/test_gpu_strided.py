"""GPU parity of strided (B, H, N, d) views: fa_fwd_strided and fa_bwd_strided.

The same values are laid out three ways that a Transformer layer produces
without copying: a (B, N, H, d) projection output transposed to (B, H, N, d);
slices of one fused (B, N, 3, H, d) QKV buffer; and rows padded past d.  Each
strided call must give the results of the contiguous call on the same values
(the kernels and their tiles are the same; only the addresses differ) and
match the fp64 oracle.  Outputs written through a view must leave the gaps of
that view untouched.
"""
import math

import numpy as np
import pytest

import oracle
from tiled_attention_04_gb300 import inputs
from test_gpu_parity import TOL, assert_close, forced_dq, oracle_all, same_dq

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def as_layout(x, B, H, layout, slot=0, pad=8):
    """The (B*H, N, d) contiguous tensor x, copied into a buffer of the given layout
    and returned as a (B, H, N, d) view of it (plus the buffer)."""
    torch = _torch()
    BH, N, d = x.shape
    x4 = x.view(B, H, N, d)
    if layout == "bhnd":
        return x4, x4
    if layout == "bnhd":   # (B, N, H, d) buffer, viewed transposed
        buf = x4.transpose(1, 2).contiguous()
        return buf.transpose(1, 2), buf
    if layout == "qkv":    # slot `slot` of a (B, N, 3, H, d) buffer
        buf = torch.zeros(B, N, 3, H, d, dtype=x.dtype, device=x.device)
        buf[:, :, slot] = x4.transpose(1, 2)
        return buf[:, :, slot].transpose(1, 2), buf
    if layout == "padded":  # rows of d + pad elements, the tail unused
        buf = torch.full((B, H, N, d + pad), 3.0, dtype=x.dtype, device=x.device)
        buf[..., :d] = x4
        return buf[..., :d], buf
    raise ValueError(layout)


def run_both(t, B, H, causal, layout, out_layout=None):
    """Contiguous call and strided call on the same values; both as numpy dicts."""
    torch = _torch()
    from tiled_attention_04_gb300 import binding
    dev = torch.device("cuda")
    Q, K, V, dO = (inputs.to_torch(x, dev) for x in t)
    BH, Nq, d = Q.shape
    Nk = K.shape[1]
    # contiguous reference call
    O, L = binding.fa_fwd(Q, K, V, is_causal=causal)
    dQ, dK, dV = binding.fa_bwd(Q, K, V, O, dO, L, is_causal=causal)
    flat = {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV}
    # strided call
    q, _ = as_layout(Q, B, H, layout, 0)
    k, _ = as_layout(K, B, H, layout, 1)
    v, _ = as_layout(V, B, H, layout, 2)
    g, _ = as_layout(dO, B, H, "bnhd" if layout == "qkv" else layout)
    o_buf = None
    if out_layout is None:
        o = None
    else:
        o, o_buf = as_layout(torch.zeros_like(Q), B, H, out_layout)
    o, l4 = binding.fa_fwd(q, k, v, is_causal=causal, O=o)
    dq, dk, dv = binding.fa_bwd(q, k, v, o, g, l4, is_causal=causal)
    torch.cuda.synchronize()
    assert binding.fa_get_device_status() == binding.FA_OK
    if out_layout == "padded":
        assert (o_buf[..., d:].float() == 3.0).all(), "write into the gaps of a padded O"
    strided = {"O": o.reshape(BH, Nq, d), "L": l4.reshape(BH, Nq), "dQ": dq.reshape(BH, Nq, d),
               "dK": dk.reshape(BH, Nk, d), "dV": dv.reshape(BH, Nk, d)}
    to_np = lambda m: {k_: v_.double().cpu().numpy() for k_, v_ in m.items()}   # noqa: E731
    return to_np(flat), to_np(strided), (q, o, dq)


CASES = [
    # B, H, N, d, dtype, causal, layout           (tensor-core path: bf16 and N >= 128)
    (2, 3, 256, 64, "bf16", True, "bnhd"),
    (2, 3, 200, 128, "bf16", False, "bnhd"),
    (1, 4, 333, 64, "bf16", True, "qkv"),
    (2, 2, 384, 128, "bf16", True, "qkv"),
    (3, 2, 256, 64, "bf16", False, "padded"),
    (1, 2, 1152, 128, "bf16", True, "bnhd"),     # long rows: work split over a CTA pair
    (4, 40, 256, 64, "bf16", True, "bnhd"),      # many short units: persistent CTAs
    (2, 3, 256, 32, "bf16", True, "bnhd"),       # head dims below 64 on the tensor cores
    (1, 2, 300, 16, "bf16", False, "qkv"),
    # fp32: split bf16 pairs on the tensor cores (N >= 128, every head dim), the
    # CUDA-core kernels below one tile, and a bf16 shape shorter than one 128-row tile
    (2, 3, 130, 32, "f32", True, "bnhd"),
    (2, 2, 256, 128, "f32", True, "qkv"),
    (1, 3, 300, 128, "f32", False, "padded"),
    (1, 3, 100, 64, "f32", False, "qkv"),
    (2, 2, 96, 16, "bf16", True, "padded"),
]


@pytest.mark.parametrize("B,H,N,d,dt,causal,layout", CASES)
def test_strided_matches_contiguous_and_oracle(cuda_lib, B, H, N, d, dt, causal, layout):
    t = inputs.make_custom(B * H, N, N, d, dt, seed=3000 + B * H + N + d)
    flat, strided, _ = run_both(t, B, H, causal, layout)
    for k in ("O", "L", "dK", "dV"):
        assert np.array_equal(flat[k], strided[k]), f"{k}: strided differs from contiguous ({layout})"
    # dQ by reduction adds fp32 partials in a run-dependent order (one bf16 step at most)
    assert same_dq(flat["dQ"], strided["dQ"]), f"dQ: strided differs from contiguous ({layout})"
    assert_close(strided, oracle_all(t, causal, 1.0 / math.sqrt(d)), TOL[dt],
                 f"B={B} H={H} N={N} d={d} {dt} causal={causal} {layout}")


@pytest.mark.parametrize("d,dt", [(64, "bf16"), (32, "f32")])
def test_output_layout_follows_query_and_padded_output(cuda_lib, d, dt):
    t = inputs.make_custom(2 * 4, 256, 256, d, dt, seed=41 + d)
    flat, strided, (q, o, dq) = run_both(t, 2, 4, True, "bnhd")
    assert o.stride() == q.stride(), "O should keep the (B, N, H, d) order of a transposed Q"
    assert dq.stride() == q.stride(), "dQ should be laid out like Q"
    flat2, strided2, _ = run_both(t, 2, 4, True, "bnhd", out_layout="padded")
    for k in ("O", "L"):
        assert np.array_equal(flat2[k], strided2[k]), k


def test_transformer_layer_qkv_projection_without_copies(cuda_lib):
    """An xl-shaped attention block (d_model 1600 = 25 heads of 64, N 256): the fused
    QKV projection is viewed as Q, K, V with no reshape copy; the gradients of x
    and of the weights equal those of the same block fed contiguous copies, and
    the attention's output and the gradients of its inputs match the oracle on
    the exact bf16 values the block produced."""
    torch = _torch()
    from tiled_attention_04_gb300 import binding
    from tiled_attention_04_gb300.autograd import flash_attention
    dev = torch.device("cuda")
    B, N, H, d = 2, 256, 25, 64
    D = H * d
    x0 = torch.from_numpy(inputs.normal(5, 0, (B, N, D))).to(dev, torch.bfloat16)
    w0 = torch.from_numpy(inputs.uniform(5, 1, (D, 3 * D), -math.sqrt(6 / (4 * D)), math.sqrt(6 / (4 * D))))
    w0 = w0.to(dev, torch.bfloat16)
    g0 = torch.from_numpy(inputs.normal(5, 2, (B, N, D))).to(dev, torch.bfloat16)
    seen = {}

    def block(copies):
        x = x0.clone().requires_grad_(True)
        w = w0.clone().requires_grad_(True)
        qkv = (x @ w).view(B, N, 3, H, d)
        q, k, v = (qkv[:, :, i].transpose(1, 2) for i in range(3))
        if copies:
            q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        else:
            assert all(binding.accepts_view(z) for z in (q, k, v))
            for z in (q, k, v):
                z.retain_grad()
        o = flash_attention(q, k, v, is_causal=True)
        if not copies:
            seen.update(q=q, k=k, v=v, o=o)
            o.register_hook(lambda grad: seen.__setitem__("dO", grad.detach().clone()))
        y = o.transpose(1, 2).reshape(B, N, D)
        y.backward(g0)
        return y.detach(), x.grad, w.grad

    with forced_dq(binding.FA_DQ_SEPARATE_PASS):   # bit-reproducible dQ, so dx and dW compare exactly
        a, b = block(False), block(True)
    for name, u, w in zip(("y", "dx", "dW"), a, b):
        assert torch.equal(u, w), f"{name} differs between the strided and the copied block"
    block(False)   # the library's own choice of dQ strategy, compared with the oracle below
    f64 = lambda z: z.detach().double().cpu().numpy().reshape(B * H, N, d)   # noqa: E731
    Q, K, V, dO = f64(seen["q"]), f64(seen["k"]), f64(seen["v"]), f64(seen["dO"])
    dQ, dK, dV, O, L, _ = oracle.attn_bwd_ref(Q, K, V, dO, 1.0 / math.sqrt(d), True)
    got = {"O": f64(seen["o"]), "L": L, "dQ": f64(seen["q"].grad), "dK": f64(seen["k"].grad),
           "dV": f64(seen["v"].grad)}
    assert_close(got, {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV}, 2e-2, "xl block, strided views")
