"""First-order bound on the bf16 backward's rounding error in dQ and dK.

Test infrastructure.  The bf16 backward of problem flash_backward forms
D = rowsum(dO * O) from the forward's stored (bf16) O, and rounds
dS = P * (dP - D) to bf16 before the two tensor-core products that use it
(dQ = scale dS K, dK = scale dS^T Q); every other step accumulates in fp32.
The bound below propagates exactly those two roundings, elementwise, through
the oracle's own fp64 P, O, D and dS.  tests/test_oracle.py checks on the CPU
that a model of the two roundings stays inside it and that planted mistakes
(D dropped, a second factor of scale) land outside it.
"""
import numpy as np

import oracle

U_BF16 = 2.0 ** -8   # unit roundoff of bf16 (8 significant bits, round to nearest)


def rounding_bound(t, causal, scale, exact_d=False):
    """Elementwise first-order bound on |dQ - dQ_exact| and |dK - dK_exact| from
    the two bf16 roundings of the backward, with u the bf16 unit roundoff:

      D_i   from the stored O (bf16):   |dD_i| <= u * sum_c |dO_ic O_ic|
      dS_ij = P_ij (dP_ij - D_i) rounded to bf16 for the MMAs, so
            |d dS_ij| <= (1 + u) P_ij |dD_i| + u |dS_ij|
      dQ_ic = scale sum_j dS_ij K_jc:  |d dQ_ic| <= scale sum_j |d dS_ij| |K_jc|
      dK_jc = scale sum_i dS_ij Q_ic:  |d dK_jc| <= scale sum_i |d dS_ij| |Q_ic|

    P, O, D and dS are the oracle's (fp64).  The fp32 terms (exp2, accumulation,
    L) are orders of magnitude smaller and covered by a 1e-3 floor in the test.
    exact_d: D formed from the unrounded O (the fused forward + backward call).
    """
    Q, K, V, dO = (x.exact for x in t)
    _, _, _, O, _, D = oracle.attn_bwd_ref(Q, K, V, dO, scale, causal)
    EQ, EK = np.empty_like(Q), np.empty_like(K)
    for b in range(Q.shape[0]):
        P, _ = oracle.attn_probs_ref(Q[b], K[b], scale, causal)
        dS = P * (dO[b] @ V[b].T - D[b][:, None])
        dD = np.zeros_like(D[b]) if exact_d else U_BF16 * np.abs(dO[b] * O[b]).sum(axis=1)
        err_dS = (1 + U_BF16) * P * dD[:, None] + U_BF16 * np.abs(dS)
        EQ[b] = scale * (err_dS @ np.abs(K[b]))
        EK[b] = scale * (err_dS.T @ np.abs(Q[b]))
    return EQ, EK
