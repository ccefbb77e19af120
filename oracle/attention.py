"""Plain fp64 CPU oracle for exact softmax attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code, header, table or
helper with the CUDA library; the two meet only on the seeded inputs.

What it computes is the definition the FlashAttention pages start from, with
every intermediate materialised in fp64 and nothing blocked, fused or
reordered:

* forward -- «把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战»,
  §一 (the three-line definition ``S = Q K^T * scale``, ``P = softmax(S)``,
  ``O = P V``).  Tiling and the online softmax of the same section reach this
  result exactly up to rounding, so the oracle is the untiled definition.
* backward -- same article, §二 (``Delta = rowsum(O * dO)``, ``P`` recomputed,
  ``dP = dO V^T``, ``dS = scale * P * (dP - Delta)``, ``dQ = dS K``,
  ``dK = dS^T Q``, ``dV = P^T dO``).
* causal -- same article, §一 (the causal bullet) and §八: the upper triangle
  (key index j > query index i) takes no part, i.e. it is masked to -inf
  before the softmax.

Readings where the pages are silent (each is listed in the design doc):

* ``lse`` is the natural-log log-sum-exp of the *scaled* scores of each row,
  ``lse_i = log(sum_j exp(S_ij))``.  The pages only say the backward
  recomputes P (§二); the saved row statistic has to be something from which
  ``P_ij = exp(S_ij - lse_i)``, and this is the plainest one.
* ``scale`` is the float32 value handed to the GPU, widened to fp64.
* Layout ``[Z, H, N, D]``; every (z, h) pair is an independent head.

Parity pins: every function here is pinned by ``tests/test_oracle.py`` against
closed forms, invariants, brute force, central finite differences and the
fp64 CPU ``torch.nn.functional.scaled_dot_product_attention`` (an independent
library).  No function is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "scores",
    "softmax_probs",
    "attn_fwd_ref",
    "attn_bwd_ref",
    "attn_fwd_head",
    "attn_bwd_head",
    "causal_tile_count",
]


def _f64(x) -> np.ndarray:
    """Exact widening of fp16/bf16/fp32 host data (numpy or torch CPU) to fp64."""
    if hasattr(x, "detach"):  # torch tensor: go through numpy without torch math
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()  # exact: every bf16 value is an fp32 value (numpy has no bf16)
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def _scale64(scale: float) -> float:
    # The GPU receives ``scale`` as a C float; the oracle uses that exact value.
    return float(np.float32(scale))


def scores(q_h: np.ndarray, k_h: np.ndarray, scale: float, causal: bool) -> np.ndarray:
    """S = Q K^T * scale for one head, with -inf above the diagonal if causal.

    §一 of «把 FlashAttention 搬上昇腾»; the mask follows §八 (upper triangle,
    key j > query i, does not take part).
    """
    s = (q_h @ k_h.T) * _scale64(scale)
    if causal:
        n_q, n_k = s.shape
        mask = np.arange(n_k)[None, :] > np.arange(n_q)[:, None]
        s = np.where(mask, -np.inf, s)
    return s


def softmax_probs(s: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Row softmax of S with its natural-log log-sum-exp.

    Returns ``(P, lse)``: ``P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i)``
    with ``m_i = max_j S_ij`` (the max subtraction only keeps exp finite; the
    value is the textbook softmax) and ``lse_i = m_i + log(sum_j exp(S_ij - m_i))``.
    """
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    l = np.sum(e, axis=1, keepdims=True)
    p = e / l
    lse = (m + np.log(l))[:, 0]
    return p, lse


def attn_fwd_head(q_h, k_h, v_h, causal: bool, scale: float):
    """Forward for one head: ``O = softmax(Q K^T scale) V`` and its lse (§一)."""
    q_h, k_h, v_h = _f64(q_h), _f64(k_h), _f64(v_h)
    p, lse = softmax_probs(scores(q_h, k_h, scale, causal))
    o = p @ v_h
    return o, lse


def attn_bwd_head(q_h, k_h, v_h, do_h, causal: bool, scale: float):
    """Backward for one head, following the equations of §二 in their order.

    ``Delta`` is taken as ``rowsum(P * dP)``, which equals ``rowsum(O * dO)``
    exactly (``O = P V`` so ``sum_d O_id dO_id = sum_j P_ij (dO V^T)_ij``);
    the test-suite checks the two agree.
    """
    q_h, k_h, v_h, do_h = _f64(q_h), _f64(k_h), _f64(v_h), _f64(do_h)
    sc = _scale64(scale)
    p, _ = softmax_probs(scores(q_h, k_h, scale, causal))
    dp = do_h @ v_h.T
    delta = np.sum(p * dp, axis=1, keepdims=True)
    ds = sc * p * (dp - delta)
    dq = ds @ k_h
    dk = ds.T @ q_h
    dv = p.T @ do_h
    return dq, dk, dv


def attn_fwd_ref(q, k, v, causal: bool, scale: float, heads=None):
    """Forward over ``[Z, H, N, D]`` inputs.  Returns fp64 ``(O, lse)``.

    ``heads``: optional iterable of flat head indices ``z * H + h``; when given
    only those heads are computed and the result has shape ``[len(heads), N, D]``
    / ``[len(heads), N]`` (used to sample the full-size workloads).
    """
    z, h, n, d = q.shape
    qf = q.reshape(z * h, n, d)
    kf = k.reshape(z * h, n, d)
    vf = v.reshape(z * h, n, d)
    idx = range(z * h) if heads is None else list(heads)
    o = np.empty((len(idx), n, d))
    lse = np.empty((len(idx), n))
    for out_i, hi in enumerate(idx):
        o[out_i], lse[out_i] = attn_fwd_head(qf[hi], kf[hi], vf[hi], causal, scale)
    if heads is None:
        return o.reshape(z, h, n, d), lse.reshape(z, h, n)
    return o, lse


def attn_bwd_ref(q, k, v, do, causal: bool, scale: float, heads=None):
    """Backward over ``[Z, H, N, D]`` inputs.  Returns fp64 ``(dQ, dK, dV)``.

    ``heads`` has the same meaning as in :func:`attn_fwd_ref`.
    """
    z, h, n, d = q.shape
    flat = [t.reshape(z * h, n, d) for t in (q, k, v, do)]
    idx = range(z * h) if heads is None else list(heads)
    outs = [np.empty((len(idx), n, d)) for _ in range(3)]
    for out_i, hi in enumerate(idx):
        g = attn_bwd_head(*(t[hi] for t in flat), causal, scale)
        for o_arr, g_arr in zip(outs, g):
            o_arr[out_i] = g_arr
    if heads is None:
        return tuple(o.reshape(z, h, n, d) for o in outs)
    return tuple(outs)


def causal_tile_count(n_tiles: int, causal: bool) -> int:
    """Number of (query tile, key tile) pairs a tiled pass visits.

    §八 of «把 FlashAttention 搬上昇腾»: with the score split into T x T tiles a
    non-causal pass visits T*T tiles and a causal pass only the lower triangle
    including the diagonal, 1 + 2 + ... + T.
    """
    if not causal:
        return n_tiles * n_tiles
    return sum(range(1, n_tiles + 1))
