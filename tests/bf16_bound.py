"""First-order bound on the bf16 backward's rounding error in dQ and dK.

Test infrastructure.  With bf16 inputs the method rounds three things to bf16
that reach dQ and dK: P before O = P V in the forward (flash_forward casts P
to V's dtype), the stored O from which the backward forms D = rowsum(dO * O)
(problem flash_backward), and dS = P * (dP - D) before the two tensor-core
products that use it (dQ = scale dS K, dK = scale dS^T Q); every other step
accumulates in fp32.  The bound below propagates exactly those roundings,
elementwise, through the oracle's own fp64 P, O, D and dS.  tests/test_oracle.py
checks on the CPU that a model of the roundings stays inside it and that
planted mistakes (D dropped, a second factor of scale) land outside it.
"""
import numpy as np

import oracle

U_BF16 = 2.0 ** -8   # unit roundoff of bf16 (8 significant bits, round to nearest)


def rounding_bound(t, causal, scale, o_rounded=True):
    """Elementwise first-order bound on |dQ - dQ_exact| and |dK - dK_exact| from
    the bf16 roundings of the method, with u the bf16 unit roundoff:

      O      the forward rounds P to bf16 before O = P V (flash_forward), so the
             fp32 O carries |dO_ic| <= u * sum_j P_ij |V_jc|; the stored O is
             that, rounded to bf16 (o_rounded): another u * |O_ic|;
      D_i    = sum_c dO_ic O_ic from that O:
             |dD_i| <= u * sum_c |dO_ic| (sum_j P_ij |V_jc| + [o_rounded] |O_ic|)
      dS_ij  = P_ij (dP_ij - D_i) rounded to bf16 for the MMAs, so
             |d dS_ij| <= (1 + u) P_ij |dD_i| + u |dS_ij|
      dQ_ic  = scale sum_j dS_ij K_jc:  |d dQ_ic| <= scale sum_j |d dS_ij| |K_jc|
      dK_jc  = scale sum_i dS_ij Q_ic:  |d dK_jc| <= scale sum_i |d dS_ij| |Q_ic|

    P, O, D and dS are the oracle's (fp64).  The fp32 terms (exp2, accumulation,
    L) are orders of magnitude smaller and covered by a 1e-3 floor in the test.
    o_rounded: D formed from the stored bf16 O (fa_bwd), else from the forward's
    fp32 O (the fused forward + backward call).
    """
    Q, K, V, dO = (x.exact for x in t)
    _, _, _, O, _, D = oracle.attn_bwd_ref(Q, K, V, dO, scale, causal)
    EQ, EK = np.empty_like(Q), np.empty_like(K)
    for b in range(Q.shape[0]):
        P, _ = oracle.attn_probs_ref(Q[b], K[b], scale, causal)
        dS = P * (dO[b] @ V[b].T - D[b][:, None])
        o_err = P @ np.abs(V[b]) + (np.abs(O[b]) if o_rounded else 0.0)
        dD = U_BF16 * (np.abs(dO[b]) * o_err).sum(axis=1)
        err_dS = (1 + U_BF16) * P * dD[:, None] + U_BF16 * np.abs(dS)
        EQ[b] = scale * (err_dS @ np.abs(K[b]))
        EK[b] = scale * (err_dS.T @ np.abs(Q[b]))
    return EQ, EK
