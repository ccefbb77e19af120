"""fp64 CPU oracle for attention over a paged K/V cache.

TEST INFRASTRUCTURE ONLY, like ``oracle/attention.py``: only the test-suite,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs use it, and it shares
nothing with the CUDA library.

Source: «把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战», the
contest section's ReshapeAndCache and GQA Paged Attention parts:

* the cache is organised in physical blocks of ``block_size`` tokens; token
  slot ``s`` lives in block ``s // block_size`` at offset ``s % block_size``;
  a negative slot means "skip this token";
* attention reads the cache through ``block_tables`` (logical block of a
  sequence -> physical block), uses ``context_lens`` for the real length of
  each sequence and masks the invalid tokens of the last block;
* query heads are an integer multiple of the K/V heads (grouped heads, as
  in ``oracle/attention.py``);
* the Quest Sparse Attention part: only a chosen subset of a sequence's
  blocks gets exact attention (``sparse_attn_fwd_ref``; how the blocks are
  chosen -- the scoring and Top-K -- is an input here).

Readings where the pages are silent: the cache layout is
``[num_blocks, block_size, H_kv, D]`` (one token's K for all K/V heads is
contiguous, which is what a per-token cache write produces); the queries of
sequence b are the last ``n_q`` tokens of its ``context_lens[b]`` tokens, so
the causal rule is the bottom-right one of ``oracle/attention.py``.

Once the cache is gathered back into a contiguous ``[H_kv, n_k, D]`` K and V,
the result is exactly the dense attention of ``oracle/attention.py``, which
this module calls.
"""

from __future__ import annotations

import numpy as np

from . import attention as dense

__all__ = ["reshape_and_cache", "gather_sequence", "paged_attn_fwd_ref", "sparse_attn_fwd_ref"]


def reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache):
    """Write new tokens into the paged cache in place (the ReshapeAndCache rule).

    ``k_new``, ``v_new``: ``[T, H_kv, D]``; ``slot_mapping``: ``[T]`` ints;
    ``k_cache``, ``v_cache``: numpy ``[num_blocks, block_size, H_kv, D]``.
    Token i goes to block ``slot // block_size``, offset ``slot % block_size``;
    tokens with a negative slot are skipped.
    """
    block_size = k_cache.shape[1]
    for i, slot in enumerate(np.asarray(slot_mapping)):
        slot = int(slot)
        if slot < 0:
            continue
        k_cache[slot // block_size, slot % block_size] = np.asarray(k_new[i])
        v_cache[slot // block_size, slot % block_size] = np.asarray(v_new[i])


def gather_sequence(cache, block_table_row, n_tokens: int) -> np.ndarray:
    """Tokens 0 .. n_tokens-1 of one sequence as ``[H_kv, n_tokens, D]`` fp64.

    Logical token p is in logical block ``p // block_size``, physical block
    ``block_table_row[p // block_size]``, offset ``p % block_size``.
    """
    cache = dense._f64(cache)
    block_size = cache.shape[1]
    rows = [cache[int(block_table_row[p // block_size]), p % block_size] for p in range(n_tokens)]
    return np.stack(rows, axis=1) if rows else np.zeros((cache.shape[2], 0, cache.shape[3]))


def paged_attn_fwd_ref(q, k_cache, v_cache, block_table, context_lens, causal: bool, scale: float):
    """Forward over ``q`` ``[B, H, n_q, D]`` and a paged cache.  Returns fp64
    ``(O [B, H, n_q, D], lse [B, H, n_q])``.

    Sequence b attends to its first ``context_lens[b]`` cached tokens; with
    ``causal`` its queries are the last ``n_q`` of them.
    """
    q = dense._f64(q)
    B, H, n_q, D = q.shape
    table = np.asarray(block_table)
    lens = np.asarray(context_lens)
    o = np.empty((B, H, n_q, D))
    lse = np.empty((B, H, n_q))
    for b in range(B):
        n_k = int(lens[b])
        k_b = gather_sequence(k_cache, table[b], n_k)[None]
        v_b = gather_sequence(v_cache, table[b], n_k)[None]
        o[b:b + 1], lse[b:b + 1] = dense.attn_fwd_ref(q[b:b + 1], k_b, v_b, causal, scale)
    return o, lse


def sparse_attn_fwd_ref(q, k_cache, v_cache, sel_pages, sel_blocks, sel_count, context_lens, causal: bool,
                        scale: float):
    """Exact attention over selected cache blocks (the contest section's
    Quest Sparse Attention: only the chosen blocks get full attention).

    For sequence b and K/V head kvh, the first ``sel_count[b, kvh]`` entries
    of ``sel_pages[b, kvh]`` / ``sel_blocks[b, kvh]`` name physical pages and
    the logical blocks they hold.  Row r of logical block L is the token at
    position ``L * block_size + r``; it takes part iff that position is below
    ``context_lens[b]`` and, when causal, at most the query's own position
    (queries are the last n_q tokens of the context).  A query row with no
    such token gets O = 0 and lse = -inf (an empty softmax).
    Returns fp64 ``(O [B, H, n_q, D], lse [B, H, n_q])``.
    """
    q = dense._f64(q)
    kc, vc = dense._f64(k_cache), dense._f64(v_cache)
    B, H, n_q, D = q.shape
    bs, h_kv = kc.shape[1], kc.shape[2]
    g = H // h_kv
    sc = dense._scale64(scale)
    pages, blocks, counts = np.asarray(sel_pages), np.asarray(sel_blocks), np.asarray(sel_count)
    lens = np.asarray(context_lens)
    o = np.zeros((B, H, n_q, D))
    lse = np.full((B, H, n_q), -np.inf)
    for b in range(B):
        n_k = int(lens[b])
        for h in range(H):
            kvh = h // g
            keys, vals, pos = [], [], []
            for e in range(int(counts[b, kvh])):
                for r in range(bs):
                    keys.append(kc[int(pages[b, kvh, e]), r, kvh])
                    vals.append(vc[int(pages[b, kvh, e]), r, kvh])
                    pos.append(int(blocks[b, kvh, e]) * bs + r)
            if not keys:
                continue
            keys, vals, pos = np.array(keys), np.array(vals), np.array(pos)
            for i in range(n_q):
                limit = (i + n_k - n_q) if causal else (n_k - 1)
                visible = (pos < n_k) & (pos <= limit)
                if not visible.any():
                    continue
                s = (keys[visible] @ q[b, h, i]) * sc
                p, l = dense.softmax_probs(s[None, :])
                o[b, h, i] = p[0] @ vals[visible]
                lse[b, h, i] = l[0]
    return o, lse
