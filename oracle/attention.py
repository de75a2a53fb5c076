"""fp64 CPU oracle for exact (Flash)attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg use it.  It shares no code with the CUDA path.

What it computes.  FlashAttention-2 is exact attention reorganised for the
memory hierarchy (CS336 A2 field guide "Systems and Parallelism", §1.2-1.3,
problems flash_forward and flash_backward; the algorithm is Dao 2023,
"FlashAttention-2").  So the oracle is the plain definition, not the tiled
algorithm:

  S   = scale * Q K^T                               (flash_forward (a))
  S  += -1e6 where key index > query index          (flash_forward (c): add, not assign)
  P   = softmax_rows(S),  L = m + ln(l)             (flash_forward (a): the saved logsumexp)
  O   = P V
  D   = rowsum(dO * O)                              (flash_backward)
  dV  = P^T dO,  dP = dO V^T,  dS = P * (dP - D)    (flash_backward)
  dQ  = scale * dS K,  dK = scale * dS^T Q          (flash_backward: one scale factor each)

Readings of points the pages leave open: natural log in L; the diagonal is
visible (mask iff key > query, top-left aligned when Nq != Nk); scale multiplies
S before the mask.

Memory.  S is materialised one block of query rows at a time, each row block
holding complete key rows, so softmax is unchanged; dK and dV are summed over
row blocks.  There is no other blocking, fusion or reordering.

Inputs are (BH, Nq, d) / (BH, Nk, d) arrays (any float dtype, upcast to fp64).
Pinned by tests/test_oracle.py: finite differences, softmax row sums, scipy's
logsumexp, torch's fp64 scaled_dot_product_attention, causal invariance, the
D identity, closed forms and a hand-worked example.
"""
from __future__ import annotations

import numpy as np

MASK_ADD = -1.0e6   # the handout's masking constant (flash_forward (c))


def _scores(Qb, K, scale, is_causal, row0):
    """S rows [row0, row0+len(Qb)) for one (batch*head): scale*Q K^T (+ mask)."""
    S = scale * (Qb @ K.T)
    if is_causal:
        qi = np.arange(row0, row0 + Qb.shape[0])[:, None]
        kj = np.arange(K.shape[0])[None, :]
        S = S + np.where(kj > qi, MASK_ADD, 0.0)
    return S


def _softmax_stats(S):
    m = S.max(axis=1)
    E = np.exp(S - m[:, None])
    l = E.sum(axis=1)
    P = E / l[:, None]
    L = m + np.log(l)
    return P, L


def attn_probs_ref(Q, K, scale, is_causal):
    """P (Nq, Nk) and L (Nq,) for ONE head: small inputs only (materialises S)."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    S = _scores(Q, K, scale, is_causal, 0)
    return _softmax_stats(S)


def attn_fwd_ref(Q, K, V, scale, is_causal, row_block=1024):
    """O (BH,Nq,d) and L (BH,Nq), fp64."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    BH, Nq, d = Q.shape
    O = np.empty((BH, Nq, V.shape[2]))
    L = np.empty((BH, Nq))
    for b in range(BH):
        for r0 in range(0, Nq, row_block):
            r1 = min(Nq, r0 + row_block)
            P, Lb = _softmax_stats(_scores(Q[b, r0:r1], K[b], scale, is_causal, r0))
            O[b, r0:r1] = P @ V[b]
            L[b, r0:r1] = Lb
    return O, L


def attn_bwd_ref(Q, K, V, dO, scale, is_causal, row_block=1024):
    """dQ, dK, dV (fp64) plus the forward's O, L and D = rowsum(dO*O).

    The backward is the closed form of flash_backward: P is rebuilt from the
    scores, D from the fp64 O, then the five matrix expressions.
    """
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    dO = np.asarray(dO, np.float64)
    BH, Nq, d = Q.shape
    Nk = K.shape[1]
    dQ = np.empty_like(Q)
    dK = np.zeros((BH, Nk, d))
    dV = np.zeros((BH, Nk, V.shape[2]))
    O = np.empty((BH, Nq, V.shape[2]))
    L = np.empty((BH, Nq))
    D = np.empty((BH, Nq))
    for b in range(BH):
        for r0 in range(0, Nq, row_block):
            r1 = min(Nq, r0 + row_block)
            P, Lb = _softmax_stats(_scores(Q[b, r0:r1], K[b], scale, is_causal, r0))
            Ob = P @ V[b]
            dOb = dO[b, r0:r1]
            Db = (dOb * Ob).sum(axis=1)
            dV[b] += P.T @ dOb
            dP = dOb @ V[b].T
            dS = P * (dP - Db[:, None])
            dQ[b, r0:r1] = scale * (dS @ K[b])
            dK[b] += scale * (dS.T @ Q[b, r0:r1])
            O[b, r0:r1] = Ob
            L[b, r0:r1] = Lb
            D[b, r0:r1] = Db
    return dQ, dK, dV, O, L, D


def attn_rows_ref(Q, K, V, dO, scale, is_causal, bh, rows):
    """O, L, D and dQ for selected query rows of one (batch*head).

    Each row depends only on its own scores, so this is the same definition
    restricted to those rows (used to check full-size outputs by sampling).
    """
    Q = np.asarray(Q[bh], np.float64)
    K = np.asarray(K[bh], np.float64)
    V = np.asarray(V[bh], np.float64)
    dO = np.asarray(dO[bh], np.float64)
    rows = np.asarray(rows)
    S = scale * (Q[rows] @ K.T)
    if is_causal:
        S = S + np.where(np.arange(K.shape[0])[None, :] > rows[:, None], MASK_ADD, 0.0)
    P, L = _softmax_stats(S)
    O = P @ V
    D = (dO[rows] * O).sum(axis=1)
    dP = dO[rows] @ V.T
    dS = P * (dP - D[:, None])
    dQ = scale * (dS @ K)
    return O, L, D, dQ


def attn_key_cols_ref(Q, K, V, dO, scale, is_causal, bh, cols, L, D):
    """dK and dV for selected key rows of one (batch*head).

    Column j of P needs every query's L and D (from this oracle's own forward);
    then dV_j = sum_i P_ij dO_i and dK_j = scale * sum_i dS_ij Q_i.
    """
    Q = np.asarray(Q[bh], np.float64)
    K = np.asarray(K[bh], np.float64)
    V = np.asarray(V[bh], np.float64)
    dO = np.asarray(dO[bh], np.float64)
    cols = np.asarray(cols)
    St = scale * (K[cols] @ Q.T)                        # (ncols, Nq) = S[:, cols]^T
    if is_causal:
        St = St + np.where(cols[:, None] > np.arange(Q.shape[0])[None, :], MASK_ADD, 0.0)
    Pt = np.exp(St - np.asarray(L[bh], np.float64)[None, :])
    dPt = V[cols] @ dO.T
    dSt = Pt * (dPt - np.asarray(D[bh], np.float64)[None, :])
    dV = Pt @ dO
    dK = scale * (dSt @ Q)
    return dK, dV
