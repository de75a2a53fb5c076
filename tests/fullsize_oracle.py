"""Every output element of a full-size workload from the fp64 oracle, on all host cores.

Test infrastructure (imported by the GPU parity tests only).  Each query row
of attention depends only on K, V and its own scores, so the oracle's row
function (O, L, D and dQ of selected query rows) runs on chunks of rows; the
key function (dK and dV of selected keys, given every query's L and D) then
runs on chunks of keys.  Both are the plain definition restricted to those
rows or keys, and both are pinned against the whole-matrix oracle in
tests/test_oracle.py.  The chunks run in a pool of *spawned* processes (never
forked: the parent may already hold a CUDA context), each regenerating the
workload's seeded inputs itself, with one BLAS thread per process.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_STATE = {}


def _init(name, dtype):
    from tiled_attention_04_gb300 import inputs
    w = inputs.WORKLOADS[name]
    t = inputs.make_inputs(w, dtype)
    _STATE["x"] = tuple(x.exact for x in t)
    _STATE["w"] = w


def _rows(task):
    import oracle
    bh, r0, r1 = task
    Q, K, V, dO = _STATE["x"]
    w = _STATE["w"]
    O, L, D, dQ = oracle.attn_rows_ref(Q, K, V, dO, w.scale, w.causal, bh, np.arange(r0, r1))
    return bh, r0, r1, O, L, D, dQ


def _keys(task):
    import oracle
    bh, c0, c1, Lrow, Drow = task
    Q, K, V, dO = _STATE["x"]
    w = _STATE["w"]
    # the key function reads L[bh] and D[bh]: hand it this head's rows at index bh
    Ls = {bh: Lrow}
    Ds = {bh: Drow}
    dK, dV = oracle.attn_key_cols_ref(Q, K, V, dO, w.scale, w.causal, bh, np.arange(c0, c1), Ls, Ds)
    return bh, c0, c1, dK, dV


def _chunk(n, bh):
    """Rows per task: about 2^25 score elements (256 MiB of fp64) at most, at least 64 rows."""
    return max(64, min(n, (1 << 25) // max(n, 1)))


def full_oracle(name, processes=None):
    """O, L, dQ, dK, dV (fp64, shapes (BH, N, d) / (BH, N)) of workload `name`."""
    from tiled_attention_04_gb300 import inputs
    w = inputs.WORKLOADS[name]
    BH, N, d = w.BH, w.N, w.d
    procs = processes or max(1, min(os.cpu_count() or 1, 32))
    ch = _chunk(N, BH)
    row_tasks = [(b, r0, min(N, r0 + ch)) for b in range(BH) for r0 in range(0, N, ch)]
    out = {"O": np.empty((BH, N, d)), "L": np.empty((BH, N)), "dQ": np.empty((BH, N, d)),
           "dK": np.empty((BH, N, d)), "dV": np.empty((BH, N, d))}
    D = np.empty((BH, N))
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(procs, initializer=_init, initargs=(name, w.dtype)) as pool:
            for b, r0, r1, O, L, Db, dQ in pool.imap_unordered(_rows, row_tasks):
                out["O"][b, r0:r1], out["L"][b, r0:r1], D[b, r0:r1], out["dQ"][b, r0:r1] = O, L, Db, dQ
            key_tasks = [(b, c0, min(N, c0 + ch), out["L"][b], D[b]) for b in range(BH) for c0 in range(0, N, ch)]
            for b, c0, c1, dK, dV in pool.imap_unordered(_keys, key_tasks):
                out["dK"][b, c0:c1], out["dV"][b, c0:c1] = dK, dV
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return out
