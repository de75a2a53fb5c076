"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such callers (code handed raw pointers by a host framework with no allocator
of its own, or code that must not call cudaMalloc/cudaFree because they can
synchronise the device) get the scratch from a fixed array inside the library
instead of a workspace argument.  It runs the same kernels as fa_bwd, so these
tests call it through the C ABI and require the results of fa_bwd (bit for bit;
for dQ formed by reduction, to one bf16 rounding step, as between two fa_bwd runs),
twice in a row on different inputs, after a larger call has left its own data
in the shared scratch, and on an empty shape; plus the refusal of unsupported
arguments and of a shape that needs more scratch than the array holds.  This file is
collected last so that a failure here cannot hide another test's result.
"""
import pytest

from tiled_attention_04_gb300 import inputs

pytestmark = pytest.mark.gpu


def t_q(t, dev, i=0):
    return inputs.to_torch(t[i], dev)


def _both(torch, binding, t, causal):
    dev = torch.device("cuda")
    Q, K, V, dO = (inputs.to_torch(x, dev) for x in t)
    O, L = binding.fa_fwd(Q, K, V, is_causal=causal)
    ref = binding.fa_bwd(Q, K, V, O, dO, L, is_causal=causal)
    got = binding.fa_bwd_noalloc(Q, K, V, O, dO, L, is_causal=causal)
    torch.cuda.synchronize()
    assert binding.fa_get_device_status() == binding.FA_OK
    return got, ref


@pytest.mark.parametrize("bh,n,d,dt,causal", [(2, 1024, 128, "bf16", True), (3, 200, 64, "bf16", False),
                                              (1, 128, 16, "f32", True), (2, 512, 128, "f32", False)])
def test_noalloc_matches_fa_bwd_twice(cuda_lib, bh, n, d, dt, causal):
    import torch
    from tiled_attention_04_gb300 import binding
    dev = torch.device("cuda")
    # a larger call first, so that the scratch holds another problem's rows
    big = inputs.make_custom(4, 2048, 2048, 64, "bf16", seed=30)
    _both(torch, binding, big, True)
    for seed in (31, 32):   # two calls in a row, different inputs
        t = inputs.make_custom(bh, n, n, d, dt, seed=seed)
        got, ref = _both(torch, binding, t, causal)
        for name, g, r in zip(("dK", "dV"), got[1:], ref[1:]):
            assert torch.equal(g, r), f"{name} differs from fa_bwd (seed {seed})"
        # dQ formed by reduction adds fp32 partial sums in a run-dependent order, so two
        # runs may differ by one bf16 rounding step; the separate pass is bit-exact
        a, b = got[0].double(), ref[0].double()
        if binding.dq_strategy(t_q(t, dev), t_q(t, dev, 1), causal) == binding.FA_DQ_SEPARATE_PASS:
            assert torch.equal(a, b), f"dQ differs from fa_bwd (seed {seed})"
        else:
            big = max(a.abs().max().item(), b.abs().max().item())
            assert bool(((a - b).abs() <= 2.0 ** -7 * torch.maximum(a.abs(), b.abs()) + 2.0 ** -16 * big).all()), \
                f"dQ (seed {seed})"


def test_noalloc_falls_back_to_the_separate_dq_pass_when_the_accumulator_does_not_fit(cuda_lib):
    """16 heads of 4096 causal query rows at d = 64: fa_bwd forms dQ by reduction,
    whose fp32 accumulator (16 MiB) exceeds the 8 MiB array; the no-alloc call
    forms dQ by the separate pass instead (no accumulator) and gives fa_bwd's
    results: dK and dV bit for bit, dQ to one bf16 rounding step."""
    import torch
    from tiled_attention_04_gb300 import binding
    t = inputs.make_custom(16, 4096, 4096, 64, "bf16", seed=33)
    Q, K = t_q(t, torch.device("cuda")), t_q(t, torch.device("cuda"), 1)
    assert binding.dq_strategy(Q, K, True) == binding.FA_DQ_REDUCTION
    assert binding.fa_bwd_workspace_size(Q, K, True) > binding.lib().fa_noalloc_scratch_bytes()
    got, ref = _both(torch, binding, t, True)
    for name, g, r in zip(("dK", "dV"), got[1:], ref[1:]):
        assert torch.equal(g, r), name
    a, b = got[0].double(), ref[0].double()
    big = max(a.abs().max().item(), b.abs().max().item())
    assert bool(((a - b).abs() <= 2.0 ** -7 * torch.maximum(a.abs(), b.abs()) + 2.0 ** -16 * big).all())


def test_noalloc_empty_queries_zero_gradients(cuda_lib):
    """No query rows: dK and dV are exactly zero and dQ is empty."""
    import torch
    from tiled_attention_04_gb300 import binding
    dev = torch.device("cuda")
    Q = torch.empty(2, 0, 64, device=dev, dtype=torch.bfloat16)
    K = torch.randn(2, 96, 64, device=dev).to(torch.bfloat16)
    L = torch.empty(2, 0, device=dev)
    dQ, dK, dV = binding.fa_bwd_noalloc(Q, K, K, Q, Q, L, is_causal=False)
    torch.cuda.synchronize()
    assert binding.fa_get_device_status() == binding.FA_OK
    assert dQ.numel() == 0 and (dK == 0).all() and (dV == 0).all()


def test_noalloc_unsupported_arguments_named_like_fa_bwd(cuda_lib):
    """Arguments fa_bwd refuses (here head dim 48) need no scratch size; the call
    reports the same status fa_bwd would, and launches nothing."""
    from tiled_attention_04_gb300 import binding
    L = binding.lib()
    assert L.fa_bwd_workspace_size(1, 2, 128, 128, 48, 0, binding.FA_DTYPE_BF16) == 0
    st = L.fa_bwd_noalloc(None, None, None, None, None, None, None, None, None, 1, 2, 128, 128, 48, 0.125, 0,
                          binding.FA_DTYPE_BF16, None)
    assert st == 3   # FA_ERR_UNSUPPORTED_HEAD_DIM


def test_noalloc_refuses_oversized_shape(cuda_lib):
    from tiled_attention_04_gb300 import binding
    L = binding.lib()
    cap = int(L.fa_noalloc_scratch_bytes())
    assert cap == 8 << 20
    # 64 heads of 65536 query rows need 2 x 4M x 4 bytes of scratch: refused before any
    # launch.  The tensor pointers are NULL, so even a regression of the size check
    # could not launch a kernel: the argument check would refuse them next.
    st = L.fa_bwd_noalloc(None, None, None, None, None, None, None, None, None, 1, 64, 65536, 65536, 64, 0.125, 1,
                          binding.FA_DTYPE_BF16, None)
    assert st == 6   # FA_ERR_WORKSPACE
