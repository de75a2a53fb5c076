"""fp32 inputs on the tensor cores: every operand split into a bf16 pair
(hi = bf16(x), lo = bf16(x - hi)) and every product of the method taken as
hi*hi + hi*lo + lo*hi with fp32 accumulation (include/fa.h, fa_set_fp32_mode);
head dims up to 64 run 128-column split rows, head dim 128 256-column ones.

At the default scale 1/sqrt(d) the outputs meet the fp32 tolerance of 1e-4
elementwise against the oracle (here on shapes of several tiles with ragged
tails, Nq != Nk, head dims 16/32/64, causal or not, and the forms the host
picks: one query tile per CTA and the two-CTA split items).  At scale 1 the
split mode is held to the first-order bound of its products (split_bound.py),
and the automatic mode takes the CUDA-core kernels there (its plain 1e-4 is
tested in test_gpu_parity.py).
"""
import math

import numpy as np
import pytest

from split_bound import split_bound, split_model
from test_gpu_parity import assert_close, oracle_all, run_gpu
from tiled_attention_04_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = [
    # bh, nq, nk, d, causal
    (2, 256, 256, 64, True), (2, 256, 256, 64, False), (3, 384, 384, 32, True), (2, 256, 256, 16, False),
    (1, 1000, 300, 64, True), (1, 300, 1000, 32, False), (3, 130, 130, 16, True), (1, 1088, 1088, 64, True),
    (1, 4096, 4096, 64, True), (8, 1024, 1024, 64, False),
    # head dim 128: 256-column split rows
    (2, 256, 256, 128, True), (2, 256, 256, 128, False), (1, 1000, 300, 128, True), (1, 300, 1000, 128, False),
    (1, 1088, 1088, 128, True), (4, 1024, 1024, 128, False),
]


@pytest.mark.parametrize("bh,nq,nk,d,causal", CASES)
def test_split_fp32_parity(cuda_lib, bh, nq, nk, d, causal):
    from tiled_attention_04_gb300 import binding
    t = inputs.make_custom(bh, nq, nk, d, "f32", seed=7000 + nq + nk + d)
    Q = inputs.to_torch(t[0])
    assert binding.path_name(nq, nk, d, causal, binding.FA_DTYPE_F32) == "tc"
    assert binding.dq_strategy(Q, inputs.to_torch(t[1]), causal) == binding.FA_DQ_SEPARATE_PASS
    got = run_gpu(t, causal)   # the default (automatic) mode at the default scale: split pairs
    assert_close(got, oracle_all(t, causal, 1.0 / math.sqrt(d)), 1e-4, f"split fp32 {bh}x{nq}x{nk} d={d}")


def test_split_fp32_modes_pick_the_kernels(cuda_lib):
    from tiled_attention_04_gb300 import binding
    f32 = binding.FA_DTYPE_F32
    with binding.fp32_mode(binding.FA_FP32_EXACT):
        assert binding.path_name(512, 512, 64, 1, f32) == "simt"
    with binding.fp32_mode(binding.FA_FP32_SPLIT):
        assert binding.path_name(512, 512, 64, 1, f32) == "tc"
        assert binding.path_name(512, 512, 128, 1, f32) == "tc"     # 256-column split rows
        assert binding.path_name(100, 512, 64, 1, f32) == "simt"    # shorter than one tile
    assert binding.path_name(512, 512, 64, 1, f32) == "tc"          # automatic, default scale
    with pytest.raises(ValueError):
        binding.set_fp32_mode(7)


def test_split_fp32_exact_mode_matches_the_cuda_core_kernels(cuda_lib):
    """FA_FP32_EXACT runs the fp32 CUDA-core kernels: the same 1e-4 from another path,
    and the two paths agree to the split path's accuracy."""
    from tiled_attention_04_gb300 import binding
    t = inputs.make_custom(2, 256, 256, 64, "f32", seed=7100)
    want = oracle_all(t, True, 0.125)
    split = run_gpu(t, True)
    with binding.fp32_mode(binding.FA_FP32_EXACT):
        exact = run_gpu(t, True)
    assert_close(exact, want, 1e-4, "exact fp32")
    assert_close(split, exact, 2e-4, "split against exact")


@pytest.mark.parametrize("d", [64, 128])
def test_split_fp32_scale_one_within_the_product_bound(cuda_lib, d):
    """Forced split mode at scale 1: scores of standard deviation sqrt(d), where the
    products' 3 * 2^-16 relative error reaches the outputs through the softmax;
    every output stays inside the first-order bound of those products, and within
    twice the errors of the numerical model of that arithmetic."""
    from tiled_attention_04_gb300 import binding
    t = inputs.make_custom(2, 256, 256, d, "f32", seed=7200 + d)
    with binding.fp32_mode(binding.FA_FP32_SPLIT):
        got = run_gpu(t, True, scale=1.0)
    want = oracle_all(t, True, 1.0)
    bound = split_bound(t, True, 1.0)
    model = split_model(t, True, 1.0)
    for k in ("O", "L", "dQ", "dK", "dV"):
        err = np.abs(got[k] - want[k])
        allowed = bound[k] + 1e-5 * (1.0 + np.abs(want[k]))   # fp32 exp2 and accumulation
        assert (err <= allowed).all(), f"{k}: max err {err.max():.3g}, worst err/bound {(err / allowed).max():.3g}"
        # and no worse than the split arithmetic itself (the bound is a worst case over signs)
        model_err = np.abs(model[k] - want[k]).max()
        assert err.max() <= 2 * model_err + 1e-5 * (1.0 + np.abs(want[k]).max()), (k, err.max(), model_err)


@pytest.mark.parametrize("d", [64, 128])
def test_split_fp32_phases_and_fused_call(cuda_lib, d):
    """The exported phases one by one, and fa_fwd_bwd, give fa_fwd + fa_bwd's
    results bit for bit (the same split copies and kernels)."""
    import torch
    from tiled_attention_04_gb300 import binding
    t = inputs.make_custom(2, 640, 640, d, "f32", seed=7300 + d)
    dev = torch.device("cuda")
    Q, K, V, dO = (inputs.to_torch(x, dev) for x in t)
    O, L = binding.fa_fwd(Q, K, V, is_causal=True)
    dQ, dK, dV = binding.fa_bwd(Q, K, V, O, dO, L, is_causal=True)
    ws = binding.alloc_workspace(Q, K, True)
    pq, pk, pv = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    binding.fa_bwd_preprocess(O, dO, L, Q, K, True, ws)
    binding.fa_bwd_dkdv(Q, K, V, dO, L, pq, pk, pv, True, ws)
    binding.fa_bwd_dq(Q, K, V, dO, L, pq, True, ws)
    fO, fL, fdQ, fdK, fdV = binding.fa_fwd_bwd(Q, K, V, dO, is_causal=True)
    torch.cuda.synchronize()
    assert binding.fa_get_device_status() == binding.FA_OK
    for name, a, b in (("dQ", pq, dQ), ("dK", pk, dK), ("dV", pv, dV), ("O", fO, O), ("L", fL, L),
                       ("fused dQ", fdQ, dQ), ("fused dK", fdK, dK), ("fused dV", fdV, dV)):
        assert torch.equal(a, b), name
    got = {k: v.double().cpu().numpy() for k, v in (("O", O), ("L", L), ("dQ", dQ), ("dK", dK), ("dV", dV))}
    assert_close(got, oracle_all(t, True, 1.0 / math.sqrt(d)), 1e-4, f"split fp32 two calls d={d}")


def test_split_fp32_deterministic(cuda_lib):
    t = inputs.make_custom(1, 2048, 2048, 64, "f32", seed=7400)
    a = run_gpu(t, True)
    b = run_gpu(t, True)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("scale", [0.125, 1.0])
def test_fp32_phases_whichever_kernels_the_scale_picks(cuda_lib, scale):
    """The preprocessing phase has no scale argument, so for fp32 inputs it prepares
    both paths' data; the later phases then take the split pairs (scale 1/8) or the
    CUDA-core kernels (scale 1, automatic mode), and match fa_bwd bit for bit."""
    import torch
    from tiled_attention_04_gb300 import binding
    t = inputs.make_custom(2, 384, 384, 64, "f32", seed=7500)
    dev = torch.device("cuda")
    Q, K, V, dO = (inputs.to_torch(x, dev) for x in t)
    O, L = binding.fa_fwd(Q, K, V, is_causal=True, scale=scale)
    dQ, dK, dV = binding.fa_bwd(Q, K, V, O, dO, L, is_causal=True, scale=scale)
    ws = binding.alloc_workspace(Q, K, True)
    pq, pk, pv = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    binding.fa_bwd_preprocess(O, dO, L, Q, K, True, ws)
    binding.fa_bwd_dkdv(Q, K, V, dO, L, pq, pk, pv, True, ws, scale=scale)
    binding.fa_bwd_dq(Q, K, V, dO, L, pq, True, ws, scale=scale)
    gq, gk, gv = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    binding.fa_bwd_grads(Q, K, V, dO, L, gq, gk, gv, True, ws, scale=scale)
    torch.cuda.synchronize()
    assert binding.fa_get_device_status() == binding.FA_OK
    for name, a, b in (("dQ", pq, dQ), ("dK", pk, dK), ("dV", pv, dV), ("grads dQ", gq, dQ), ("grads dK", gk, dK),
                       ("grads dV", gv, dV)):
        assert torch.equal(a, b), name
    got = {k: v.double().cpu().numpy() for k, v in (("O", O), ("L", L), ("dQ", dQ), ("dK", dK), ("dV", dV))}
    assert_close(got, oracle_all(t, True, scale), 1e-4, f"fp32 phases scale={scale}")
