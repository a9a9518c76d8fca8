"""Per-expert oracle GEMMs on a process pool (test infrastructure).

The oracle's grouped GEMMs are independent per expert; at the prefill sizes
the tests run every expert, so the experts go to a pool of spawned worker
processes (spawned, not forked: the parent holds a CUDA context).  Each
worker runs the oracle function itself on one expert's rows and weights with
a single BLAS thread; nothing here computes any step of the method.
"""

from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _gmm1_one(args):
    from oracle import moe
    xq, xs, wq, ws, I = args
    return moe.gmm1_swiglu_quant(xq, xs, wq[None], ws[None], np.array([0, xq.shape[0]]), I)


def _gmm2_one(args):
    from oracle import moe
    aq, as_, wq, ws = args
    return moe.gmm2(aq, as_, wq[None], ws[None], np.array([0, aq.shape[0]]))


def _pool_map(fn, items):
    saved = {v: os.environ.get(v) for v in _BLAS_VARS}
    for v in _BLAS_VARS:
        os.environ[v] = "1"
    try:
        workers = max(1, min(16, os.cpu_count() or 1, len(items)))
        with mp.get_context("spawn").Pool(workers) as pool:
            return pool.map(fn, items, chunksize=1)
    finally:
        for v, val in saved.items():
            if val is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = val


def gmm1_all_experts(xq, xs, w13q, w13s, offsets, I):
    """oracle gmm1 (SwiGLU + requant) on every non-empty expert; rows of
    empty experts stay zero, as in the oracle's own loop."""
    experts = [e for e in range(w13q.shape[0]) if offsets[e + 1] > offsets[e]]
    items = [(xq[offsets[e]:offsets[e + 1]], xs[offsets[e]:offsets[e + 1]], w13q[e], w13s[e], I)
             for e in experts]
    aq = np.zeros((xq.shape[0], I), np.uint8)
    as_ = np.zeros((xq.shape[0], I // 32), np.uint8)
    for e, (a_q, a_s) in zip(experts, _pool_map(_gmm1_one, items)):
        aq[offsets[e]:offsets[e + 1]] = a_q
        as_[offsets[e]:offsets[e + 1]] = a_s
    return aq, as_


def gmm2_all_experts(aq, as_, w2q, w2s, offsets):
    """oracle gmm2 (bf16 bits) on every non-empty expert."""
    experts = [e for e in range(w2q.shape[0]) if offsets[e + 1] > offsets[e]]
    items = [(aq[offsets[e]:offsets[e + 1]], as_[offsets[e]:offsets[e + 1]], w2q[e], w2s[e])
             for e in experts]
    y = np.zeros((aq.shape[0], w2q.shape[1]), np.uint16)
    for e, y_e in zip(experts, _pool_map(_gmm2_one, items)):
        y[offsets[e]:offsets[e + 1]] = y_e
    return y
