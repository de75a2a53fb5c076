"""Failure detection without a GPU fault: a host switch makes the forward's
MMA issuer wait on a barrier that nothing arrives on; with a small poll cap the
bounded wait gives up, the kernel reports FA_ERR_TIMEOUT through
fa_get_device_status and returns.  The context stays usable and the next call
(switch off, default cap) is correct again."""
import math

import numpy as np
import pytest

import oracle
from tiled_attention_04_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_forced_wait_timeout_reports_and_recovers(cuda_lib):
    import torch
    from tiled_attention_04_gb300 import binding
    dev = torch.device("cuda")
    t = inputs.make_custom(2, 512, 512, 128, "bf16", seed=21)
    Q, K, V, dO = (inputs.to_torch(x, dev) for x in t)
    assert binding.path_name(512, 512, 128, 1, binding.FA_DTYPE_BF16) == "tc"
    binding.fa_reset_device_status()
    try:
        binding.fa_set_wait_limit(1000)
        binding.fa_debug_force_stall(True)
        binding.fa_fwd(Q, K, V, is_causal=True)
        assert binding.fa_get_device_status() == 8      # FA_ERR_TIMEOUT
    finally:
        binding.fa_debug_force_stall(False)
        binding.fa_set_wait_limit(0)
    binding.fa_reset_device_status()
    assert binding.fa_get_device_status() == binding.FA_OK
    O, L = binding.fa_fwd(Q, K, V, is_causal=True)
    torch.cuda.synchronize()
    assert binding.fa_get_device_status() == binding.FA_OK
    rO, rL = oracle.attn_fwd_ref(t[0].exact, t[1].exact, t[2].exact, 1 / math.sqrt(128), True)
    np.testing.assert_allclose(O.double().cpu().numpy(), rO, rtol=2e-2, atol=2e-2)
    np.testing.assert_allclose(L.double().cpu().numpy(), rL, rtol=2e-2, atol=2e-2)


def test_forced_wait_timeout_in_persistent_forward(cuda_lib):
    """The same failure path in the persistent forward (many short query tiles:
    320 batch*heads of 256 rows), whose softmax warpgroups hand results over
    through mbarriers between work units."""
    import torch
    from tiled_attention_04_gb300 import binding
    dev = torch.device("cuda")
    t = inputs.make_custom(320, 256, 256, 64, "bf16", seed=22)
    Q, K, V, dO = (inputs.to_torch(x, dev) for x in t)
    binding.fa_reset_device_status()
    try:
        binding.fa_set_wait_limit(1000)
        binding.fa_debug_force_stall(True)
        binding.fa_fwd(Q, K, V, is_causal=True)
        assert binding.fa_get_device_status() == 8      # FA_ERR_TIMEOUT
    finally:
        binding.fa_debug_force_stall(False)
        binding.fa_set_wait_limit(0)
    binding.fa_reset_device_status()
    O, L = binding.fa_fwd(Q, K, V, is_causal=True)
    torch.cuda.synchronize()
    assert binding.fa_get_device_status() == binding.FA_OK
    rO, rL = oracle.attn_fwd_ref(t[0].exact, t[1].exact, t[2].exact, 1 / math.sqrt(64), True)
    np.testing.assert_allclose(O.double().cpu().numpy(), rO, rtol=2e-2, atol=2e-2)
    np.testing.assert_allclose(L.double().cpu().numpy(), rL, rtol=2e-2, atol=2e-2)
