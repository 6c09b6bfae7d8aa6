"""The fp64 oracle over every segment of a large workload, segments spread
over a pool of host processes (attention is block-diagonal, so each
segment's scores and LSE depend on that segment alone).

Test infrastructure: it only calls oracle.importance segment by segment and
puts the pieces back in place. The pool uses the spawn start method, so it
is safe after the parent process has initialised CUDA."""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def _segment(args):
    import oracle
    qb, kb, nq, nk, scale, fmt = args
    return oracle.importance(qb, kb, [0, nq], [0, nk], scale, fmt=fmt)


def importance_by_segment(w, softmax_scale=None, fmt="bf16", workers=None):
    """(lse [H, Tq], scores [Tk]) of oracle.importance over the whole workload."""
    cq, ck = np.asarray(w.cu_seqlens_q), np.asarray(w.cu_seqlens_k)
    G = len(ck) - 1
    tasks = []
    for g in range(G):
        q0, q1, k0, k1 = int(cq[g]), int(cq[g + 1]), int(ck[g]), int(ck[g + 1])
        tasks.append((w.q_bits[q0:q1], w.k_bits[k0:k1], q1 - q0, k1 - k0, softmax_scale, fmt))
    # longest first, so the pool does not end on one large segment
    order = sorted(range(G), key=lambda g: -(tasks[g][2] * tasks[g][3]))
    workers = workers or os.cpu_count() or 1
    saved = {v: os.environ.get(v) for v in _BLAS_VARS}
    for v in _BLAS_VARS:
        os.environ[v] = "1"   # one BLAS thread per process (inherited by the spawned workers)
    try:
        with cf.ProcessPoolExecutor(max_workers=min(workers, max(G, 1)),
                                    mp_context=mp.get_context("spawn")) as ex:
            results = dict(zip(order, ex.map(_segment, [tasks[g] for g in order])))
    finally:
        for v, x in saved.items():
            if x is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = x
    H = w.q_bits.shape[1]
    lse = np.full((H, int(cq[-1])), -np.inf)
    scores = np.zeros(int(ck[-1]))
    for g in range(G):
        l_g, s_g = results[g]
        lse[:, int(cq[g]):int(cq[g + 1])] = l_g
        scores[int(ck[g]):int(ck[g + 1])] = s_g
    return lse, scores
