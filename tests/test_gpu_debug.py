"""The debug build (libfa_debug.so, compiled with FA_DEBUG) on small shapes.

Its kernels check every tile they load against the tensor's extent and, under
the causal mask, against the diagonal (a failed check records FA_ERR_BOUNDS,
skips the access and ends the kernel's waits; it never traps), and they count
the tile rows they load.  These tests run the whole forward + backward through
it and require: no failed check; exactly the tiles at or below the diagonal
loaded (the counts of the method's causal early exit, field guide §1.3.3); the
release library's results (bit for bit where its results are reproducible);
and the oracle's.
"""
import math

import numpy as np
import pytest

from test_gpu_parity import assert_close, forced_dq, oracle_all, same_dq
from tiled_attention_04_gb300 import inputs

pytestmark = pytest.mark.gpu


def _cdiv(a, b):
    return (a + b - 1) // b


def expected_rows(bh, nq, nk, d, causal, reduction, narrow=False):
    """Tile rows the tensor-core kernels must load, by the loops of the method:
    forward   every 128-row query tile loads the 128-key tiles up to its last
              visible key;
    dK/dV     every 128-key tile loads the query sub-tiles (128 rows; 64 at
              d = 128) from the one holding its first key's row to the end;
    dQ        every 128-row query tile loads the key sub-tiles (128 / 64 rows)
              up to its last visible key (none when dQ is formed by reduction).
    narrow: fp32 split into bf16 pairs, which runs the 64-wide d = 128 items
    (32-wide for head dim 128, whose split rows are 256 columns)."""
    if narrow:
        sub = 32 if d == 128 else 64
    else:
        sub = 64 if d == 128 else 128
    fwd = kv = dq = 0
    for qt in range(_cdiv(nq, 128)):
        kend = min(nk, qt * 128 + 128) if causal else nk
        fwd += _cdiv(kend, 128) * 128
        dq += _cdiv(kend, sub) * sub
    for kt in range(_cdiv(nk, 128)):
        first = (kt * 128) // sub if causal else 0
        kv += max(0, _cdiv(nq, sub) - first) * sub
    return [bh * fwd, bh * kv, 0 if reduction else bh * dq]


CASES = [
    # bh, nq, nk, d, causal
    (2, 512, 512, 64, True), (1, 1088, 1088, 64, True), (3, 384, 384, 64, False), (1, 200, 333, 64, True),
    (1, 333, 200, 64, True), (2, 1152, 1152, 128, True), (2, 640, 640, 128, False), (1, 300, 1000, 128, True),
    (2, 333, 129, 32, False), (1, 1152, 1152, 16, True),
    (320, 256, 256, 64, True), (1, 4096, 4096, 64, True), (1, 4096, 4096, 128, True),
]


def _run(t, causal, call):
    import torch
    from tiled_attention_04_gb300 import binding
    dev = torch.device("cuda")
    Q, K, V, dO = (inputs.to_torch(x, dev) for x in t)
    if call == "fused":
        out = binding.fa_fwd_bwd(Q, K, V, dO, is_causal=causal)
    else:
        O, L = binding.fa_fwd(Q, K, V, is_causal=causal)
        out = (O, L) + tuple(binding.fa_bwd(Q, K, V, O, dO, L, is_causal=causal))
    torch.cuda.synchronize()
    return {k: v.double().cpu().numpy() for k, v in zip(("O", "L", "dQ", "dK", "dV"), out)}


@pytest.mark.parametrize("bh,nq,nk,d,causal", CASES)
@pytest.mark.parametrize("call", ["fused", "two_calls"])
def test_debug_build_loads_exactly_the_visible_tiles(cuda_lib, bh, nq, nk, d, causal, call):
    import torch
    from tiled_attention_04_gb300 import binding
    t = inputs.make_custom(bh, nq, nk, d, "bf16", seed=6000 + bh + nq + nk + d)
    Q = inputs.to_torch(t[0], torch.device("cuda"))
    K = inputs.to_torch(t[1], torch.device("cuda"))
    release = _run(t, causal, call)
    red = binding.dq_strategy(Q, K, causal) == binding.FA_DQ_REDUCTION
    with binding.debug_library() as D:
        assert D.fa_debug_build() == 1
        binding.fa_reset_device_status()
        binding.debug_reset_tile_rows()
        got = _run(t, causal, call)
        status = binding.fa_get_device_status()
        rows = binding.debug_tile_rows()
    assert status == binding.FA_OK, binding.STATUS.get(status, status)
    assert rows == expected_rows(bh, nq, nk, d, causal, red), (rows, expected_rows(bh, nq, nk, d, causal, red))
    for k in ("O", "L", "dK", "dV"):
        assert np.array_equal(got[k], release[k]), f"{k}: debug build differs from the release build"
    assert same_dq(got["dQ"], release["dQ"])
    assert_close(got, oracle_all(t, causal, 1.0 / math.sqrt(d)), 2e-2, f"debug build {call} {bh}x{nq}x{nk} d={d}")


def test_debug_build_counts_the_separate_dq_pass(cuda_lib):
    """Forced separate dQ pass at d = 64: the dQ items' key rows are counted too."""
    from tiled_attention_04_gb300 import binding
    t = inputs.make_custom(2, 640, 640, 64, "bf16", seed=6100)
    with binding.debug_library():
        # the strategy is a setting of each library: force it in the debug library
        with forced_dq(binding.FA_DQ_SEPARATE_PASS):
            binding.fa_reset_device_status()
            binding.debug_reset_tile_rows()
            got = _run(t, True, "two_calls")
            status = binding.fa_get_device_status()
            rows = binding.debug_tile_rows()
    assert status == binding.FA_OK
    assert rows == expected_rows(2, 640, 640, 64, True, False)
    assert_close(got, oracle_all(t, True, 1 / 8), 2e-2, "debug build, separate dQ pass")


def test_release_build_counts_nothing(cuda_lib):
    from tiled_attention_04_gb300 import binding
    t = inputs.make_custom(1, 256, 256, 64, "bf16", seed=6200)
    _run(t, True, "fused")
    assert binding.lib().fa_debug_build() == 0
    assert binding.debug_tile_rows() == [0, 0, 0]


@pytest.mark.parametrize("bh,nq,nk,d,causal", [(2, 512, 512, 64, True), (1, 300, 1000, 32, False),
                                               (1, 2048, 2048, 64, True), (2, 640, 640, 128, True),
                                               (1, 333, 777, 128, False)])
def test_debug_build_split_fp32(cuda_lib, bh, nq, nk, d, causal):
    """fp32 split into bf16 pairs (the d = 128 kernels on 128-column copies): no failed
    check, the visible tiles' rows exactly, the release library's results bit for bit
    (dQ by the separate pass) and the oracle's at 1e-4."""
    from tiled_attention_04_gb300 import binding
    t = inputs.make_custom(bh, nq, nk, d, "f32", seed=6300 + nq + d)
    release = _run(t, causal, "two_calls")
    with binding.debug_library() as D:
        assert D.fa_debug_build() == 1
        binding.fa_reset_device_status()
        binding.debug_reset_tile_rows()
        got = _run(t, causal, "fused")
        status = binding.fa_get_device_status()
        rows = binding.debug_tile_rows()
    assert status == binding.FA_OK, binding.STATUS.get(status, status)
    assert rows == expected_rows(bh, nq, nk, d, causal, False, narrow=True)
    for k in got:
        assert np.array_equal(got[k], release[k]), k
    assert_close(got, oracle_all(t, causal, 1.0 / math.sqrt(d)), 1e-4, f"debug split fp32 {bh}x{nq}x{nk}")
