"""Writes tests/golden/samples_<workload>.npz: oracle values at sampled rows of the full-size workloads.

Calls only the oracle (oracle/) and the seeded input generator.  For each
sampled (batch*head) it runs the oracle over every query row (in chunks) to get
L and D, keeps O, L and dQ at the sampled query rows, then evaluates dK and dV
at the sampled key rows from those L and D.  The input digests are stored so a
test can confirm it drew the same inputs before comparing.

Usage: python tests/golden/make_samples.py [workload ...]
"""
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from tiled_attention_04_gb300 import inputs  # noqa: E402

FULL = ["bench_b8_n4096_d64_causal", "long_n16384_d128_causal", "vlong_n65536_d64_causal",
        "layer_xl_b4_h25_n1024_causal", "layer_xl_b4_h25_n1024_full"]


def sample_rows(N, rng, k=24):
    fixed = {0, 1, 63, 64, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1}
    extra = set(rng.choice(N, size=k, replace=False).tolist())
    return np.array(sorted(r for r in fixed | extra if 0 <= r < N))


def sample_bh(BH):
    return sorted({0, BH - 1, BH // 2}) if BH > 1 else [0]


def make(name, chunk=512):
    w = inputs.WORKLOADS[name]
    t0 = time.time()
    Q, K, V, dO = inputs.make_inputs(w)
    rng = np.random.default_rng(w.seed + 1000)
    bhs = sample_bh(w.BH)
    rows = sample_rows(w.N, rng)
    cols = sample_rows(w.N, rng)
    out = {"bh": np.array(bhs), "rows": rows, "cols": cols,
           "digest": np.array([inputs.storage_digest(t) for t in (Q, K, V, dO)])}
    O_s, L_s, dQ_s, dK_s, dV_s = [], [], [], [], []
    row_set = set(rows.tolist())
    for bh in bhs:
        L_all = np.empty(w.N)
        D_all = np.empty(w.N)
        keep = {}
        for r0 in range(0, w.N, chunk):
            rr = np.arange(r0, min(w.N, r0 + chunk))
            O, L, D, dQ = oracle.attn_rows_ref(Q.exact, K.exact, V.exact, dO.exact, w.scale, w.causal, bh, rr)
            L_all[rr] = L
            D_all[rr] = D
            for i, r in enumerate(rr):
                if r in row_set:
                    keep[int(r)] = (O[i], L[i], dQ[i])
        O_s.append(np.stack([keep[int(r)][0] for r in rows]))
        L_s.append(np.array([keep[int(r)][1] for r in rows]))
        dQ_s.append(np.stack([keep[int(r)][2] for r in rows]))
        dKc, dVc = oracle.attn_key_cols_ref(Q.exact, K.exact, V.exact, dO.exact, w.scale, w.causal, bh, cols,
                                            {bh: L_all}, {bh: D_all})
        dK_s.append(dKc)
        dV_s.append(dVc)
    out.update(O=np.stack(O_s), L=np.stack(L_s), dQ=np.stack(dQ_s), dK=np.stack(dK_s), dV=np.stack(dV_s))
    path = os.path.join(HERE, f"samples_{name}.npz")
    np.savez_compressed(path, **out)
    print(f"{name}: {time.time() - t0:.1f}s -> {path}", flush=True)


if __name__ == "__main__":
    for n in (sys.argv[1:] or FULL):
        make(n)
