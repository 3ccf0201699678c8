"""Runs the fp64 oracle on full-size prefill workloads in parallel processes.

The oracle is called unchanged on pieces of the problem that are themselves
complete causal-prefill problems: the query heads of one KV head and a range
of query rows [r0, r1), whose rows sit at absolute positions q_offset + r0 ..
and see the keys 0 .. q_offset + r1 - 1 at most.  Every row's result depends
only on its own query and visible keys, so the pieces put together are the
oracle's answer for the whole problem.  The pool uses the ``spawn`` start
method (never ``fork`` after CUDA is initialised) and one BLAS thread per
worker.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _prefill_piece(args):
    import oracle
    q, k, v, q_offset, scale = args
    return oracle.prefill_causal(q, k, v, q_offset, scale)


def prefill_causal_parallel(q, k, v, q_offset, scale, workers=None, row_pieces=None):
    """oracle.prefill_causal over the whole problem, split over processes.

    q [B, H_q, T_q, d], k/v [B, H_kv, S_kv, d] as float32 or float64 numpy
    arrays (bf16 values are exact in both).  Returns O, lse in float64.
    """
    B, H_q, T_q, d = q.shape
    H_kv = k.shape[1]
    G = H_q // H_kv
    workers = workers or max(1, min(32, os.cpu_count() or 1))
    if row_pieces is None:
        row_pieces = max(1, min(T_q // 128, -(-2 * workers // (B * H_kv))))
    edges = np.linspace(0, T_q, row_pieces + 1).astype(int)
    tasks, where = [], []
    for b in range(B):
        for kv in range(H_kv):
            heads = slice(kv * G, (kv + 1) * G)
            for r0, r1 in zip(edges[:-1], edges[1:]):
                if r1 <= r0:
                    continue
                n_keys = q_offset + r1
                tasks.append((np.ascontiguousarray(q[b:b + 1, heads, r0:r1]),
                              np.ascontiguousarray(k[b:b + 1, kv:kv + 1, :n_keys]),
                              np.ascontiguousarray(v[b:b + 1, kv:kv + 1, :n_keys]),
                              q_offset + r0, scale))
                where.append((b, heads, r0, r1))
    saved = {n: os.environ.get(n) for n in _BLAS_VARS}
    for n in _BLAS_VARS:
        os.environ[n] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(min(workers, len(tasks))) as pool:
            results = pool.map(_prefill_piece, tasks, chunksize=1)
    finally:
        for n, val in saved.items():
            if val is None:
                os.environ.pop(n, None)
            else:
                os.environ[n] = val
    o = np.zeros((B, H_q, T_q, d))
    lse = np.zeros((B, H_q, T_q))
    for (b, heads, r0, r1), (po, pl) in zip(where, results):
        o[b, heads, r0:r1] = po[0]
        lse[b, heads, r0:r1] = pl[0]
    return o, lse
