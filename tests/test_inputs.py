"""The seeded input generator: published SplitMix64 outputs, bf16 rounding, workload shapes."""
import numpy as np
import pytest

from tiled_attention_04_gb300 import inputs


def test_splitmix64_matches_published_sequence():
    # SplitMix64 seeded with 0 starts 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F
    # (Steele, Lea & Flood 2014 reference generator); output k of stream s is mix(s + (k+1)*golden).
    got = [int(x) for x in inputs.splitmix64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert int(inputs.splitmix64(0, 2, 1)[0]) == 0x06C45D188009454F


def test_normal_moments_and_determinism():
    z = inputs.normal(7, 3, (200000,))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert np.array_equal(z, inputs.normal(7, 3, (200000,)))
    assert not np.array_equal(z[:100], inputs.normal(7, 4, (100,)))


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = inputs.normal(5, 1, (4096,)) * 37.0
    b = inputs.to_bf16_bits(x)
    t = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, t)
    assert np.array_equal(inputs.bf16_bits_to_f64(b), torch.from_numpy(t.view(np.int16)).view(torch.bfloat16).double().numpy())


def test_workload_shapes_and_flops():
    w = inputs.WORKLOADS["bench_b8_n4096_d64_causal"]
    assert (w.BH, w.N, w.d, w.dtype, w.causal) == (8, 4096, 64, "bf16", True)
    f, b = w.flops()
    assert f == 4 * 8 * 4096 * 4096 * 64 / 2 and b == 2.5 * f
    t = inputs.WORKLOADS["tiny_f32_causal"]
    Q, K, V, dO = inputs.make_inputs(t)
    assert Q.shape == (1, 128, 16) and Q.storage.dtype == np.float32
    assert np.array_equal(Q.exact, Q.storage.astype(np.float64))


def test_projected_layer_inputs():
    w = inputs.WORKLOADS["layer_xl_b4_h25_n1024_causal"]
    small = inputs.Workload("p", 2, 3, 8, 4, "bf16", True, 4, projected=True)
    Q, K, V, dO = inputs.make_inputs(small)
    assert Q.shape == (6, 8, 4) and Q.storage.dtype == np.uint16
    # Xavier-uniform projections of unit normals keep the per-element variance near 1
    assert w.BH == 100 and w.d == 64
