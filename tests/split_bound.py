"""First-order error bound of fp32 attention computed from split bf16 pairs.

Test infrastructure.  The split path (include/fa.h, fa_set_fp32_mode) writes
every fp32 operand x as hi = bf16(x) plus lo = bf16(x - hi) and forms every
product of the method -- S = Q K^T and O = P V (flash_forward), dP = dO V^T,
dV = P^T dO, dQ = scale dS K, dK = scale dS^T Q (flash_backward) -- as
hi*hi + hi*lo + lo*hi with fp32 accumulation.  With u = 2^-8 (bf16's unit
roundoff) x = hi + lo + r with |r| <= u^2 |x| and |lo| <= (u + u^2) |x|, so
each such sum of products x_i y_i is off by at most about e = 3 u^2 times
sum |x_i y_i| (the dropped lo*lo and the two residuals r).  The bound
propagates that, elementwise and to first order, through the oracle's fp64
P, O, D and dS:

  scores   |dS_ij|  <= e scale sum_c |Q_ic| |K_jc|
  L        |dL_i|   <= sum_j P_ij |dS_ij|              (logsumexp)
  P        |dP_ij|  <= P_ij (|dS_ij| + |dL_i|)          (forward and backward)
  O        |dO_ic|  <= sum_j |dP_ij| |V_jc| + e sum_j P_ij |V_jc|
  D        |dD_i|   <= sum_c |dO_ic| |dO_ic(O)|          (D from the fp32 O)
  dP       |d dP|   <= e sum_c |dO_ic| |V_jc|
  dS       |d dS|   <= |dP_ij| |dP - D| + P_ij (|d dP_ij| + |dD_i|)
  dV, dQ, dK: the same two terms (the error of the operand that carries one,
           plus e times the sum of the magnitudes of the products).

fp32 effects (exp2, accumulation, the stored L) are two orders of magnitude
smaller and covered by a separate floor in the tests.  split_model() is a
numerical model of the split arithmetic (fp64 sums of the split operands'
products) that the CPU tests hold inside this bound, and that planted mistakes
push outside it.
"""
import numpy as np

import oracle

U = 2.0 ** -8
E_SPLIT = 3 * U * U   # relative error of one hi*hi + hi*lo + lo*hi sum of products


def split_bound(t, causal, scale):
    """Elementwise bounds on |O - O_exact|, |L - L_exact|, |dQ - ...|, |dK - ...|, |dV - ...|."""
    Q, K, V, dO = (x.exact for x in t)
    _, _, _, O, _, D = oracle.attn_bwd_ref(Q, K, V, dO, scale, causal)
    out = {k: [] for k in ("O", "L", "dQ", "dK", "dV")}
    for b in range(Q.shape[0]):
        P, _ = oracle.attn_probs_ref(Q[b], K[b], scale, causal)
        aQ, aK, aV, adO = np.abs(Q[b]), np.abs(K[b]), np.abs(V[b]), np.abs(dO[b])
        eS = E_SPLIT * abs(scale) * (aQ @ aK.T)
        eL = (P * eS).sum(axis=1)
        eP = P * (eS + eL[:, None])
        eO = eP @ aV + E_SPLIT * (P @ aV)
        eD = (adO * eO).sum(axis=1)
        dPm = dO[b] @ V[b].T
        edP = E_SPLIT * (adO @ aV.T)
        dS = P * (dPm - D[b][:, None])
        edS = eP * np.abs(dPm - D[b][:, None]) + P * (edP + eD[:, None])
        out["O"].append(eO)
        out["L"].append(eL)
        out["dV"].append(eP.T @ adO + E_SPLIT * (P.T @ adO))
        out["dQ"].append(abs(scale) * (edS @ aK + E_SPLIT * (np.abs(dS) @ aK)))
        out["dK"].append(abs(scale) * (edS.T @ aQ + E_SPLIT * (np.abs(dS).T @ aQ)))
    return {k: np.stack(v) for k, v in out.items()}


def _bf16(x):
    """Round to bf16 (nearest, ties to even) through fp32; returns fp64."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def _split(x):
    x32 = np.asarray(x, np.float32).astype(np.float64)
    hi = _bf16(x32)
    return hi, _bf16(x32 - hi)


def _mm(a, b, terms):
    ah, al = _split(a)
    bh, bl = _split(b)
    r = ah @ bh
    if terms >= 2:
        r = r + ah @ bl
    if terms >= 3:
        r = r + al @ bh
    return r


def split_model(t, causal, scale, terms=3, drop_d=False):
    """The split arithmetic in fp64: every product from the split operands (terms = 3:
    hi hi + hi lo + lo hi; fewer terms model a kernel that drops products), P from the
    model's own scores and logsumexp, D from the model's O rounded to fp32."""
    Q, K, V, dO = (x.exact for x in t)
    out = {k: [] for k in ("O", "L", "dQ", "dK", "dV")}
    for b in range(Q.shape[0]):
        S = _mm(Q[b], K[b].T, terms) * scale
        if causal:
            S = np.where(np.tril(np.ones(S.shape, bool)), S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        p = np.exp(S - m)
        l = p.sum(axis=1, keepdims=True)
        Ob = _mm(p, V[b], terms) / l
        Ob = Ob.astype(np.float32).astype(np.float64)
        Lb = (m + np.log(l))[:, 0]
        Db = 0.0 if drop_d else (Ob * dO[b]).sum(axis=1, keepdims=True)
        P = np.exp(S - Lb[:, None])
        dS = P * (_mm(dO[b], V[b].T, terms) - Db)
        out["O"].append(Ob)
        out["L"].append(Lb)
        out["dV"].append(_mm(P.T, dO[b], terms))
        out["dQ"].append(_mm(dS, K[b], terms) * scale)
        out["dK"].append(_mm(dS.T, Q[b], terms) * scale)
    return {k: np.stack(v) for k, v in out.items()}
