"""CPU pins of the split-pair error bound (tests/split_bound.py) used by the
fp32 tensor-core tests: the split itself, a numerical model of the split
arithmetic inside the bound, and planted mistakes outside it."""
import numpy as np
import pytest

import oracle
from split_bound import U, _bf16, _split, split_bound, split_model
from tiled_attention_04_gb300 import inputs


def _oracle(t, causal, scale):
    Q, K, V, dO = (x.exact for x in t)
    dQ, dK, dV, O, L, D = oracle.attn_bwd_ref(Q, K, V, dO, scale, causal)
    return {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV}


def test_split_pair_definition():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    hi, lo = _split(x)
    xd = x.astype(np.float64)
    assert np.array_equal(hi, _bf16(hi)) and np.array_equal(lo, _bf16(lo))   # both are bf16 numbers
    assert (np.abs(xd - hi) <= U * np.abs(xd)).all()
    assert (np.abs(xd - hi - lo) <= U * U * np.abs(xd)).all()
    # bf16 rounding: 1 + 2^-8 is a tie and goes to the even neighbour 1; 1 + 3 * 2^-8 rounds up
    assert _bf16(np.float32(1 + 2.0 ** -8)) == 1.0 and _bf16(np.float32(1 + 3 * 2.0 ** -8)) == 1 + 2.0 ** -6


CASES = [(2, 96, 64, True, 0.125), (2, 96, 64, True, 1.0), (1, 80, 32, False, 32 ** -0.5), (1, 80, 32, False, 1.0)]


@pytest.mark.parametrize("bh,n,d,causal,scale", CASES)
def test_split_model_inside_bound(bh, n, d, causal, scale):
    t = inputs.make_custom(bh, n, n, d, "f32", seed=11)
    want, bound = _oracle(t, causal, scale), split_bound(t, causal, scale)
    model = split_model(t, causal, scale)
    for k in want:
        assert (np.abs(model[k] - want[k]) <= bound[k] + 1e-12).all(), k


@pytest.mark.parametrize("bh,n,d,causal,scale", CASES)
def test_planted_mistakes_leave_the_bound(bh, n, d, causal, scale):
    """Dropping a product (one or two of the three) or D breaks the bound."""
    t = inputs.make_custom(bh, n, n, d, "f32", seed=11)
    want, bound = _oracle(t, causal, scale), split_bound(t, causal, scale)
    for kw, keys in (({"terms": 1}, ("O", "L", "dQ", "dK", "dV")), ({"terms": 2}, ("O", "L", "dQ", "dK", "dV")),
                     ({"drop_d": True}, ("dQ", "dK"))):
        model = split_model(t, causal, scale, **kw)
        for k in keys:
            assert (np.abs(model[k] - want[k]) > bound[k]).any(), (kw, k)
