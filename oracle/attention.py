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
* grouped K/V heads -- same article, the GQA Paged Attention part of the
  contest section: the number of query heads is an integer multiple g of the
  number of K/V heads and several query heads share one K/V head.  Query head
  h reads K/V head ``h // g``; a shared K or V gets the sum of the gradients
  of every query head that reads it (chain rule).
* query and key lengths -- the same part: a query attends to the context of
  its sequence (``context_lens``), and the last incomplete block is masked.
  Queries and keys may have different lengths n_q and n_k, any length >= 1.

Readings where the pages are silent:

* ``lse`` is the natural-log log-sum-exp of the *scaled* scores of each row,
  ``lse_i = log(sum_j exp(S_ij))``.  The pages only say the backward
  recomputes P (§二); the saved row statistic has to be something from which
  ``P_ij = exp(S_ij - lse_i)``, and this is the plainest one.
* ``scale`` is the float32 value handed to the GPU, widened to fp64.
* Layout ``[Z, H, N, D]``; every (z, h) pair is an independent head.  With
  grouped heads, Q/O/dO are ``[Z, H, n_q, D]`` and K/V ``[Z, H_kv, n_k, D]``.
* Causal with n_q != n_k: the queries are the last n_q positions of an n_k
  long sequence (the decode reading of the contest section, where a new
  token sees its whole context), so query i sees key j iff
  ``j <= i + (n_k - n_q)``; for n_q == n_k this is §八's triangle.  n_q > n_k
  would leave the first rows with no visible key and no softmax; the pages
  never form such a row, and the oracle refuses it.

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
    "kv_head_of",
    "sampled_kv_heads",
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
    key j > query i, does not take part), with the diagonal moved to
    ``j > i + (n_k - n_q)`` when the query block is the end of a longer
    sequence (module docstring).
    """
    s = (q_h @ k_h.T) * _scale64(scale)
    if causal:
        n_q, n_k = s.shape
        if n_q > n_k:
            raise ValueError("causal attention needs n_q <= n_k (every query sees at least one key)")
        mask = np.arange(n_k)[None, :] > np.arange(n_q)[:, None] + (n_k - n_q)
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


def _group(q, k) -> int:
    """Query heads per K/V head (the GQA ratio g); K/V must divide Q's heads."""
    h, h_kv = q.shape[1], k.shape[1]
    if q.shape[0] != k.shape[0] or h % h_kv != 0 or q.shape[3] != k.shape[3]:
        raise ValueError(f"incompatible q {tuple(q.shape)} and k {tuple(k.shape)}")
    return h // h_kv


def kv_head_of(head: int, group: int) -> int:
    """Flat K/V head read by flat query head ``z * H + h``: ``z * H_kv + h // g``.

    Since ``H = g * H_kv`` this is the flat query head divided by g.
    """
    return head // group


def attn_fwd_ref(q, k, v, causal: bool, scale: float, heads=None):
    """Forward over ``[Z, H, n_q, D]`` queries and ``[Z, H_kv, n_k, D]`` keys
    and values.  Returns fp64 ``(O, lse)`` shaped like q and ``[Z, H, n_q]``.

    ``heads``: optional iterable of flat query-head indices ``z * H + h``; when
    given only those heads are computed and the result has shape
    ``[len(heads), n_q, D]`` / ``[len(heads), n_q]`` (used to sample the
    full-size workloads).
    """
    g = _group(q, k)
    z, h, n_q, d = q.shape
    n_k = k.shape[2]
    qf = q.reshape(z * h, n_q, d)
    kf = k.reshape(z * h // g, n_k, d)
    vf = v.reshape(z * h // g, n_k, d)
    idx = range(z * h) if heads is None else list(heads)
    o = np.empty((len(idx), n_q, d))
    lse = np.empty((len(idx), n_q))
    for out_i, hi in enumerate(idx):
        kv = kv_head_of(hi, g)
        o[out_i], lse[out_i] = attn_fwd_head(qf[hi], kf[kv], vf[kv], causal, scale)
    if heads is None:
        return o.reshape(z, h, n_q, d), lse.reshape(z, h, n_q)
    return o, lse


def attn_bwd_ref(q, k, v, do, causal: bool, scale: float, heads=None):
    """Backward over ``[Z, H, n_q, D]`` q, do and ``[Z, H_kv, n_k, D]`` k, v.
    Returns fp64 ``(dQ, dK, dV)`` shaped like q, k, v.

    dK and dV of a K/V head sum the per-head gradients of the g query heads
    that read it.  ``heads``: optional flat query-head indices; dQ is then
    returned for those heads (``[len(heads), n_q, D]``) and dK, dV for
    ``sampled_kv_heads(heads, g)`` (each summed over its whole group).
    """
    g = _group(q, k)
    z, h, n_q, d = q.shape
    n_k = k.shape[2]
    qf, dof = q.reshape(z * h, n_q, d), do.reshape(z * h, n_q, d)
    kf, vf = k.reshape(z * h // g, n_k, d), v.reshape(z * h // g, n_k, d)
    if heads is None:
        q_idx, kv_idx = list(range(z * h)), list(range(z * h // g))
    else:
        q_idx, kv_idx = list(heads), sampled_kv_heads(heads, g)
    dq = np.empty((len(q_idx), n_q, d))
    dk = np.zeros((len(kv_idx), n_k, d))
    dv = np.zeros((len(kv_idx), n_k, d))
    kv_pos = {kvh: i for i, kvh in enumerate(kv_idx)}
    need = sorted(set(q_idx) | {kvh * g + r for kvh in kv_idx for r in range(g)})
    for hi in need:
        kv = kv_head_of(hi, g)
        gq, gk, gv = attn_bwd_head(qf[hi], kf[kv], vf[kv], dof[hi], causal, scale)
        if hi in q_idx:
            dq[q_idx.index(hi)] = gq
        if kv in kv_pos:
            dk[kv_pos[kv]] += gk
            dv[kv_pos[kv]] += gv
    if heads is None:
        return dq.reshape(z, h, n_q, d), dk.reshape(z, h // g, n_k, d), dv.reshape(z, h // g, n_k, d)
    return dq, dk, dv


def sampled_kv_heads(heads, group: int) -> list:
    """The K/V heads read by the query heads ``heads``, in first-use order."""
    out = []
    for hi in heads:
        kv = kv_head_of(hi, group)
        if kv not in out:
            out.append(kv)
    return out


def causal_tile_count(n_tiles: int, causal: bool) -> int:
    """Number of (query tile, key tile) pairs a tiled pass visits.

    §八 of «把 FlashAttention 搬上昇腾»: with the score split into T x T tiles a
    non-causal pass visits T*T tiles and a causal pass only the lower triangle
    including the diagonal, 1 + 2 + ... + T.
    """
    if not causal:
        return n_tiles * n_tiles
    return sum(range(1, n_tiles + 1))
