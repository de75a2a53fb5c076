"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such callers (code handed raw pointers by a host framework with no allocator
of its own, or code that must not call cudaMalloc/cudaFree because they can
synchronise the device) get the scratch from a fixed array inside the library
instead of a workspace argument.  These tests call it through the C ABI and
check it against fa_bwd on the same inputs, twice in a row (the second call
finds the first call's leftovers in the shared scratch), plus the refusal of a
shape that needs more scratch than the array holds.  This file is collected
last so that a failure here cannot hide another test's result.
"""
import numpy as np
import pytest

from tiled_attention_04_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bh,n,d,dt,causal", [(2, 1024, 128, "bf16", True), (3, 200, 64, "bf16", False),
                                              (1, 128, 16, "f32", True)])
def test_noalloc_matches_fa_bwd_twice(cuda_lib, bh, n, d, dt, causal):
    import torch
    from tiled_attention_04_gb300 import binding
    dev = torch.device("cuda")
    tol = 2e-2 if dt == "bf16" else 1e-4
    outs = []
    for seed in (31, 32):   # two calls in a row, different inputs
        t = inputs.make_custom(bh, n, n, d, dt, seed=seed)
        Q, K, V, dO = (inputs.to_torch(x, dev) for x in t)
        O, L = binding.fa_fwd(Q, K, V, is_causal=causal)
        ref = binding.fa_bwd(Q, K, V, O, dO, L, is_causal=causal)
        got = binding.fa_bwd_noalloc(Q, K, V, O, dO, L, is_causal=causal)
        torch.cuda.synchronize()
        assert binding.fa_get_device_status() == binding.FA_OK
        for g, r in zip(got, ref):
            g, r = g.double().cpu().numpy(), r.double().cpu().numpy()
            assert np.allclose(g, r, rtol=tol, atol=tol)
        outs.append(got[0].double().cpu().numpy())
    assert not np.array_equal(outs[0], outs[1])


def test_noalloc_refuses_oversized_shape(cuda_lib):
    from tiled_attention_04_gb300 import binding
    L = binding.lib()
    cap = int(L.fa_noalloc_scratch_bytes())
    assert cap == 8 << 20
    # 64 heads of 65536 query rows need 2 x 4M x 4 bytes of scratch: refused before any launch
    V16 = binding.ctypes.c_void_p(256)
    st = L.fa_bwd_noalloc(V16, V16, V16, V16, V16, V16, V16, V16, V16, 1, 64, 65536, 65536, 64, 0.125, 1,
                          binding.FA_DTYPE_BF16, None)
    assert st == 6   # FA_ERR_WORKSPACE
