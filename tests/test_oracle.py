"""Pins for the fp64 oracle, each against something other than the oracle itself.

* hand-worked examples (tests/golden/worked_examples.json), derived on paper;
* central finite differences of f = sum(O * dO) on tiny inputs;
* rows of P summing to one, and exact zeros above the causal diagonal;
* L against scipy's logsumexp;
* O and all three gradients against torch's fp64 CPU scaled_dot_product_attention
  under autograd (a library special case: the -1e6 mask underflows to exactly
  the same probabilities as -inf in fp64);
* causal invariance (future keys and values do not reach earlier rows);
* the D identity rowsum(dO*O) = rowsum(P*dP) of flash_backward;
* closed forms (identical keys, identical values) and symmetries;
* planted mistakes: broken copies of the oracle must fail these pins.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as oatt
from tiled_attention_04_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, amp=1.0):
    return amp * inputs.normal(seed, 0, shape)


def _ev(s):
    return float(eval(s, {"__builtins__": {}}, {"ln": math.log}))


def _ev_arr(a):
    return np.array([[_ev(x) for x in row] for row in a]) if isinstance(a[0], list) else np.array([_ev(x) for x in a])


# --------------------------------------------------------------------------- worked examples

@pytest.mark.parametrize("causal", [False, True])
def test_worked_examples(causal):
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        ex = json.load(f)["examples"]
    for e in ex:
        sc = _ev(e["scale"])
        Q, K, V, dO = (_ev_arr(e[k])[None] for k in ("Q", "K", "V", "dO"))
        want = e["causal" if causal else "noncausal"]
        O, L = oracle.attn_fwd_ref(Q, K, V, sc, causal)
        dQ, dK, dV, O2, L2, D = oracle.attn_bwd_ref(Q, K, V, dO, sc, causal)
        np.testing.assert_allclose(O[0], _ev_arr(want["O"]), rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(L[0], _ev_arr(want["L"]), rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(D[0], _ev_arr(want["D"]), rtol=1e-14, atol=1e-14)
        for name, got in (("dQ", dQ), ("dK", dK), ("dV", dV)):
            np.testing.assert_allclose(got[0], _ev_arr(want[name]), rtol=1e-13, atol=1e-14, err_msg=name)


# --------------------------------------------------------------------------- finite differences

def _fd_check(Q, K, V, dO, scale, causal, fwd=oracle.attn_fwd_ref, bwd=oracle.attn_bwd_ref, h=1e-6):
    dQ, dK, dV = bwd(Q, K, V, dO, scale, causal)[:3]

    def f(q, k, v):
        return float((fwd(q, k, v, scale, causal)[0] * dO).sum())

    worst = 0.0
    for X, G, which in ((Q, dQ, 0), (K, dK, 1), (V, dV, 2)):
        for idx in np.ndindex(X.shape):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += h
            fp = f(*args)
            args[which][idx] -= 2 * h
            fm = f(*args)
            fd = (fp - fm) / (2 * h)
            err = abs(fd - G[idx]) / (1.0 + abs(G[idx]))
            worst = max(worst, err)
    return worst


FD_CASES = [(nq, nk, d) for nq in (1, 2, 3, 5, 8) for d in (1, 2, 4) for nk in (nq,)] + [(3, 5, 2), (5, 3, 4), (8, 2, 2)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk,d", FD_CASES)
def test_finite_differences(nq, nk, d, causal):
    seed = 100 * nq + 10 * nk + d
    Q = _rand((1, nq, d), seed)
    K = _rand((1, nk, d), seed + 1)
    V = _rand((1, nk, d), seed + 2)
    dO = _rand((1, nq, d), seed + 3)
    assert _fd_check(Q, K, V, dO, 1.0 / math.sqrt(d) if d > 1 else 0.7, causal) < 1e-6


# --------------------------------------------------------------------------- softmax, L, library

@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_and_causal_zeros(causal):
    Q = _rand((37, 16), 1)
    K = _rand((37, 16), 2)
    P, L = oracle.attn_probs_ref(Q, K, 0.25, causal)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert (P >= 0).all()
    if causal:
        assert (P[np.triu_indices(37, 1)] == 0.0).all()
        assert (P[np.diag_indices(37)] > 0).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(40, 40), (24, 56), (56, 24)])
def test_L_is_logsumexp(nq, nk, causal):
    from scipy.special import logsumexp
    Q = _rand((nq, 32), 3, 2.0)
    K = _rand((nk, 32), 4, 2.0)
    sc = 1.0 / math.sqrt(32)
    P, L = oracle.attn_probs_ref(Q, K, sc, causal)
    S = sc * Q @ K.T
    if causal:
        S = np.where(np.arange(nk)[None, :] > np.arange(nq)[:, None], -np.inf, S)
    np.testing.assert_allclose(L, logsumexp(S, axis=1), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(P, np.exp(S - L[:, None]), rtol=1e-12, atol=1e-15)


def _torch_sdpa(Q, K, V, dO, scale, causal):
    torch = pytest.importorskip("torch")
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    o.backward(torch.tensor(dO, dtype=torch.float64))
    return o.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("bh,n,d", [(2, 64, 16), (1, 200, 32), (3, 48, 64), (1, 96, 128)])
def test_matches_torch_sdpa_fp64(bh, n, d, causal):
    Q, K, V, dO = (_rand((bh, n, d), 10 + t) for t in range(4))
    sc = 1.0 / math.sqrt(d)
    O, L = oracle.attn_fwd_ref(Q, K, V, sc, causal, row_block=37)
    dQ, dK, dV, *_ = oracle.attn_bwd_ref(Q, K, V, dO, sc, causal, row_block=29)
    tO, tdQ, tdK, tdV = _torch_sdpa(Q, K, V, dO, sc, causal)
    for got, want in ((O, tO), (dQ, tdQ), (dK, tdK), (dV, tdV)):
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------- causal invariance

def test_causal_invariance_forward():
    n, d = 50, 16
    Q, K, V = (_rand((1, n, d), 20 + t) for t in range(3))
    O, L = oracle.attn_fwd_ref(Q, K, V, 0.25, True)
    for i in (0, 7, 31, 48):
        K2, V2 = K.copy(), V.copy()
        K2[0, i + 1:] += _rand((n - i - 1, d), 99 + i, 3.0)
        V2[0, i + 1:] -= _rand((n - i - 1, d), 199 + i, 3.0)
        O2, L2 = oracle.attn_fwd_ref(Q, K2, V2, 0.25, True)
        assert np.array_equal(O2[0, :i + 1], O[0, :i + 1])
        assert np.array_equal(L2[0, :i + 1], L[0, :i + 1])


def test_causal_invariance_backward():
    n, d = 50, 16
    Q, K, V, dO = (_rand((1, n, d), 30 + t) for t in range(4))
    dQ, dK, dV, *_ = oracle.attn_bwd_ref(Q, K, V, dO, 0.25, True)
    for j in (3, 20, 49):
        Q2, dO2 = Q.copy(), dO.copy()
        Q2[0, :j] += _rand((j, d), 7 + j, 2.0)
        dO2[0, :j] *= -3.0
        _, dK2, dV2, *_ = oracle.attn_bwd_ref(Q2, K, V, dO2, 0.25, True)
        np.testing.assert_allclose(dK2[0, j:], dK[0, j:], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(dV2[0, j:], dV[0, j:], rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------- identities

@pytest.mark.parametrize("causal", [False, True])
def test_D_identity(causal):
    Q, K, V, dO = (_rand((45, 8), 40 + t) for t in range(4))
    P, L = oracle.attn_probs_ref(Q, K, 0.3, causal)
    O = P @ V
    dP = dO @ V.T
    _, _, _, O2, L2, D = oracle.attn_bwd_ref(Q[None], K[None], V[None], dO[None], 0.3, causal)
    np.testing.assert_allclose(D[0], (P * dP).sum(axis=1), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O2[0], O, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_uniform_attention(causal):
    n, d = 33, 8
    Q = _rand((1, n, d), 50)
    k = _rand((d,), 51)
    K = np.broadcast_to(k, (1, n, d)).copy()
    V = _rand((1, n, d), 52)
    sc = 0.5
    O, L = oracle.attn_fwd_ref(Q, K, V, sc, causal)
    cnt = np.arange(1, n + 1) if causal else np.full(n, n)
    mean = np.cumsum(V[0], axis=0) / cnt[:, None] if causal else np.broadcast_to(V[0].mean(axis=0), (n, d))
    np.testing.assert_allclose(O[0], mean, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L[0], sc * (Q[0] @ k) + np.log(cnt), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_values_give_constant_output_and_zero_qk_grads(causal):
    n, d = 29, 4
    Q, K, dO = (_rand((1, n, d), 60 + t) for t in range(3))
    c = np.array([0.5, -1.25, 2.0, 3.0])
    V = np.broadcast_to(c, (1, n, d)).copy()
    dQ, dK, dV, O, L, D = oracle.attn_bwd_ref(Q, K, V, dO, 0.5, causal)
    np.testing.assert_allclose(O[0], np.broadcast_to(c, (n, d)), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dQ, 0.0, atol=1e-12)
    np.testing.assert_allclose(dK, 0.0, atol=1e-12)
    np.testing.assert_allclose(dV[0].sum(axis=0), dO[0].sum(axis=0), rtol=1e-12, atol=1e-12)


def test_key_permutation_symmetry():
    n, d = 31, 8
    Q, K, V, dO = (_rand((1, n, d), 70 + t) for t in range(4))
    perm = np.random.default_rng(0).permutation(n)
    dQ, dK, dV, O, L, _ = oracle.attn_bwd_ref(Q, K, V, dO, 0.4, False)
    dQ2, dK2, dV2, O2, L2, _ = oracle.attn_bwd_ref(Q, K[:, perm], V[:, perm], dO, 0.4, False)
    np.testing.assert_allclose(O2, O, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(L2, L, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dQ2, dQ, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dK2, dK[:, perm], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dV2, dV[:, perm], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_query_scale_symmetry(causal):
    Q, K, V, dO = (_rand((1, 21, 8), 80 + t) for t in range(4))
    a = 3.0
    dQ, dK, dV, O, L, _ = oracle.attn_bwd_ref(Q, K, V, dO, 0.4, causal)
    dQ2, dK2, dV2, O2, L2, _ = oracle.attn_bwd_ref(a * Q, K, V, dO, 0.4 / a, causal)
    np.testing.assert_allclose(O2, O, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L2, L, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(a * dQ2, dQ, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dK2, dK, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dV2, dV, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- samplers vs full

@pytest.mark.parametrize("causal", [False, True])
def test_row_and_column_samplers_match_full(causal):
    Q, K, V, dO = (_rand((2, 70, 16), 90 + t) for t in range(4))
    dQ, dK, dV, O, L, D = oracle.attn_bwd_ref(Q, K, V, dO, 0.25, causal)
    rows = np.array([0, 1, 17, 69])
    Or, Lr, Dr, dQr = oracle.attn_rows_ref(Q, K, V, dO, 0.25, causal, 1, rows)
    np.testing.assert_allclose(Or, O[1, rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Lr, L[1, rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Dr, D[1, rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dQr, dQ[1, rows], rtol=1e-12, atol=1e-13)
    cols = np.array([0, 5, 68, 69])
    dKc, dVc = oracle.attn_key_cols_ref(Q, K, V, dO, 0.25, causal, 0, cols, L, D)
    np.testing.assert_allclose(dKc, dK[0, cols], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dVc, dV[0, cols], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- planted mistakes

def _broken_bwd(kind):
    def bwd(Q, K, V, dO, scale, causal):
        dQ, dK, dV, O, L, D = oracle.attn_bwd_ref(Q, K, V, dO, scale, causal)
        if kind == "double_scale_dK":
            dK = dK * scale
        elif kind == "no_scale_dQ":
            dQ = dQ / scale
        elif kind == "drop_D":
            P, _ = oracle.attn_probs_ref(Q[0], K[0], scale, causal)
            dS = P * (dO[0] @ V[0].T)
            dQ = scale * (dS @ K[0])[None]
        elif kind == "transposed_dV":
            P, _ = oracle.attn_probs_ref(Q[0], K[0], scale, causal)
            dV = (P @ dO[0])[None]
        return dQ, dK, dV, O, L, D
    return bwd


@pytest.mark.parametrize("kind", ["double_scale_dK", "no_scale_dQ", "drop_D", "transposed_dV"])
def test_planted_gradient_mistakes_are_caught(kind):
    Q, K, V, dO = (_rand((1, 4, 4), 110 + t) for t in range(4))
    assert _fd_check(Q, K, V, dO, 0.5, True, bwd=_broken_bwd(kind)) > 1e-3


@pytest.mark.parametrize("mistake", ["mask_diagonal", "mask_transposed", "no_scale"])
def test_planted_mask_mistakes_are_caught(monkeypatch, mistake):
    """Break the oracle's score routine; the library pin must reject it."""
    good = oatt._scores

    def bad(Qb, K, scale, is_causal, row0):
        S = scale * (Qb @ K.T)
        qi = np.arange(row0, row0 + Qb.shape[0])[:, None]
        kj = np.arange(K.shape[0])[None, :]
        if mistake == "mask_diagonal":
            S = S + np.where(kj >= qi, oatt.MASK_ADD, 0.0) * (qi > 0)
        elif mistake == "mask_transposed":
            S = S + np.where(kj < qi, oatt.MASK_ADD, 0.0)
        elif mistake == "no_scale":
            S = good(Qb, K, 1.0, is_causal, row0)
        return S

    monkeypatch.setattr(oatt, "_scores", bad)
    Q, K, V, dO = (_rand((1, 24, 8), 120 + t) for t in range(4))
    O, _ = oracle.attn_fwd_ref(Q, K, V, 0.35, True)
    tO = _torch_sdpa(Q, K, V, dO, 0.35, True)[0]
    assert not np.allclose(O, tO, rtol=1e-6, atol=1e-6)


def test_sweep_vanilla_baseline_matches_oracle():
    """The vanilla attention the latency sweep compares against computes the same
    attention (checked here on the CPU in fp64, causal and not)."""
    torch = pytest.importorskip("torch")
    from tiled_attention_04_gb300.sweep import vanilla
    rng = np.random.default_rng(11)
    for causal in (False, True):
        Q, K, V = (rng.standard_normal((2, 1, 12, 8)) for _ in range(3))
        got = vanilla(*(torch.from_numpy(x) for x in (Q, K, V)), causal, 0.3).numpy()
        for b in range(2):
            O, L = oracle.attn_fwd_ref(Q[b], K[b], V[b], 0.3, causal)
            np.testing.assert_allclose(got[b], O, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- bf16 rounding bound

def _bf16(x):
    """Round fp64 values to bf16 (nearest even, via fp32) and back to fp64."""
    return inputs.bf16_bits_to_f64(inputs.to_bf16_bits(x))


def _rounded_backward(t, causal, scale, mistake=None, o_rounded=True):
    """dQ, dK with the bf16 roundings of the kernels modelled in fp64: P rounded
    before O = P V, D from that O (rounded to bf16 when o_rounded), dS rounded to
    bf16 before its two products.  `mistake` plants an error a kernel could make
    (on the CPU, in this model)."""
    Q, K, V, dO = (x.exact for x in t)
    dQ, dK = np.empty_like(Q), np.empty_like(K)
    for b in range(Q.shape[0]):
        P, _ = oracle.attn_probs_ref(Q[b], K[b], scale, causal)
        O = _bf16(P) @ V[b]
        if o_rounded:
            O = _bf16(O)
        D = (dO[b] * O).sum(axis=1)
        if mistake == "no_D":
            D = np.zeros_like(D)
        dS = _bf16(P * (dO[b] @ V[b].T - D[:, None]))
        s = scale * scale if mistake == "double_scale" else scale
        dQ[b] = s * (dS @ K[b])
        dK[b] = scale * (dS.T @ Q[b])
    return dQ, dK


@pytest.mark.parametrize("o_rounded", [True, False])
@pytest.mark.parametrize("scale,d", [(0.25, 64), (1.0, 64), (1.0, 16), (2.0, 128)])
def test_bf16_rounding_bound_holds_for_the_rounding_model(scale, d, o_rounded):
    """The bound used by the bf16 large-scale GPU parity tests contains the error of
    the roundings it models, at a margin (the bound is worst-case), for D from
    the stored bf16 O (fa_bwd) and from the forward's fp32 O (fused call)."""
    from bf16_bound import rounding_bound
    t = inputs.make_custom(2, 160, 160, d, "bf16", seed=60 + d)
    dQ, dK, _, _, _, _ = oracle.attn_bwd_ref(*(x.exact for x in t), scale, True)
    gQ, gK = _rounded_backward(t, True, scale, o_rounded=o_rounded)
    EQ, EK = rounding_bound(t, True, scale, o_rounded=o_rounded)
    assert (np.abs(gQ - dQ) <= EQ + 1e-12).all()
    assert (np.abs(gK - dK) <= EK + 1e-12).all()
    assert np.abs(gQ - dQ).max() > 0.05 * EQ.max()   # the bound is not vacuous


@pytest.mark.parametrize("mistake", ["no_D", "double_scale"])
def test_bf16_rounding_bound_catches_planted_mistakes(mistake):
    from bf16_bound import rounding_bound
    t = inputs.make_custom(2, 160, 160, 64, "bf16", seed=61)
    dQ, dK, _, _, _, _ = oracle.attn_bwd_ref(*(x.exact for x in t), 0.5, True)
    gQ, gK = _rounded_backward(t, True, 0.5, mistake=mistake)
    EQ, EK = rounding_bound(t, True, 0.5)
    outside = (np.abs(gQ - dQ) > EQ + 1e-3 * (1 + np.abs(dQ))).sum()
    assert outside > 0.01 * dQ.size
