"""Every-head comparison of a whole workload against the fp64 oracle, spread
over the host cores.

The oracle runs head by head (forward, then backward) in worker processes
started with ``spawn`` (a process forked after CUDA initialised can hang), each
with single-threaded BLAS.  A worker receives a chunk of heads -- the inputs
and the GPU's outputs as numpy arrays -- and returns each head's errors:

    O max-abs, lse max-abs, dQ / dK / dV relative Frobenius error

This module imports only numpy and the oracle, so a worker starts without
torch.  Grouped K/V heads are out of its scope: the workloads it serves have
one K/V head per query head.
"""

from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from oracle import attention as orc

FIELDS = ("o_max_abs", "lse_max_abs", "dq_rel_fro", "dk_rel_fro", "dv_rel_fro")


def _rel_fro(g: np.ndarray, r: np.ndarray) -> float:
    return float(np.linalg.norm(g.astype(np.float64) - r) / max(np.linalg.norm(r), 1e-30))


def _check_chunk(task):
    """Oracle for heads ``ids`` and the GPU's errors on each of them."""
    ids, q, k, v, do, o, lse, dq, dk, dv, causal, scale = task
    out = np.empty((len(ids), len(FIELDS)))
    for i in range(len(ids)):
        o_ref, lse_ref = orc.attn_fwd_head(q[i], k[i], v[i], causal, scale)
        dq_ref, dk_ref, dv_ref = orc.attn_bwd_head(q[i], k[i], v[i], do[i], causal, scale)
        out[i, 0] = float(np.max(np.abs(o[i].astype(np.float64) - o_ref)))
        out[i, 1] = float(np.max(np.abs(lse[i].astype(np.float64) - lse_ref)))
        out[i, 2] = _rel_fro(dq[i], dq_ref)
        out[i, 3] = _rel_fro(dk[i], dk_ref)
        out[i, 4] = _rel_fro(dv[i], dv_ref)
    return ids, out


def workers() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(n, 64))


def all_head_errors(q, k, v, do, o, lse, dq, dk, dv, causal: bool, scale: float, chunk: int = 8) -> np.ndarray:
    """Errors of every head, ``[heads, len(FIELDS)]``.

    Arguments are host numpy arrays: q, k, v, do, o, dq, dk, dv ``[heads, N,
    D]`` (fp16, or fp32 holding bf16 values exactly) and lse ``[heads, N]``.
    """
    heads = q.shape[0]
    tasks = []
    for h0 in range(0, heads, chunk):
        sl = slice(h0, min(h0 + chunk, heads))
        tasks.append((list(range(h0, sl.stop)), q[sl], k[sl], v[sl], do[sl], o[sl], lse[sl], dq[sl], dk[sl], dv[sl],
                      bool(causal), float(scale)))
    errs = np.full((heads, len(FIELDS)), np.nan)
    n = min(workers(), len(tasks))
    if n <= 1:
        for t in tasks:
            ids, e = _check_chunk(t)
            errs[ids] = e
        return errs
    # one BLAS thread per worker: the parallelism is over heads
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {key: os.environ.get(key) for key in keys}
    try:
        for key in keys:
            os.environ[key] = "1"
        with mp.get_context("spawn").Pool(n) as pool:
            for ids, e in pool.imap_unordered(_check_chunk, tasks):
                errs[ids] = e
    finally:
        for key, val in saved.items():
            if val is None:
                os.environ.pop(key, None)
            else:
                os.environ[key] = val
    return errs
