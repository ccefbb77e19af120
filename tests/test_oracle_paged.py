"""Pins for the paged-cache oracle (CPU only).

Checked against things other than itself: a pure-Python brute force that
reads the cache through the block/offset rule of the pages, the dense
oracle on a contiguously laid out cache (a reduction to the pinned dense
case), invariance to where the physical blocks live, indifference to the
contents of slots past a sequence's context length, and the cache-write rule
(including skipped tokens).  Planted mistakes are caught.
"""

import math

import numpy as np
import pytest

from oracle import attention as orc
from oracle import paged


def rand_cache(num_blocks, block_size, h_kv, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((num_blocks, block_size, h_kv, d)),
            rng.standard_normal((num_blocks, block_size, h_kv, d)))


def brute_paged(q, kc, vc, table, lens, causal, scale):
    """Pure-Python loops; token p of sequence b is read from physical block
    table[b][p // bs] at offset p % bs."""
    B, H, n_q, D = q.shape
    bs, h_kv = kc.shape[1], kc.shape[2]
    g = H // h_kv
    out = np.zeros(q.shape)
    for b in range(B):
        n_k = int(lens[b])
        for h in range(H):
            kvh = h // g
            for i in range(n_q):
                s = []
                for p in range(n_k):
                    if causal and p > i + n_k - n_q:
                        continue
                    blk, off = int(table[b][p // bs]), p % bs
                    s.append((blk, off, scale * sum(q[b, h, i, t] * kc[blk, off, kvh, t] for t in range(D))))
                mx = max(x for _, _, x in s)
                w = [(blk, off, math.exp(x - mx)) for blk, off, x in s]
                tot = sum(x for _, _, x in w)
                for t in range(D):
                    out[b, h, i, t] = sum(x * vc[blk, off, kvh, t] for blk, off, x in w) / tot
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_small(causal):
    rng = np.random.default_rng(1)
    kc, vc = rand_cache(7, 4, 2, 3, 2)
    table = np.array([[5, 0, 3], [2, 6, 1]])
    lens = np.array([9, 5])
    q = rng.standard_normal((2, 4, 3, 3))
    sc = float(np.float32(0.7))  # the oracle, like the GPU, uses the float32 scale
    o, _ = paged.paged_attn_fwd_ref(q, kc, vc, table, lens, causal, sc)
    np.testing.assert_allclose(o, brute_paged(q, kc, vc, table, lens, causal, sc), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_contiguous_cache_equals_dense(causal):
    # Blocks laid out in order (table row b = b*nb .. b*nb+nb-1) and every
    # sequence full: the paged result is the dense result on the same K, V.
    rng = np.random.default_rng(3)
    B, H, h_kv, n_q, n_k, D, bs = 2, 6, 3, 5, 24, 8, 8
    k = rng.standard_normal((B, h_kv, n_k, D))
    v = rng.standard_normal((B, h_kv, n_k, D))
    q = rng.standard_normal((B, H, n_q, D))
    nb = n_k // bs
    kc = k.reshape(B, h_kv, nb, bs, D).transpose(0, 2, 3, 1, 4).reshape(B * nb, bs, h_kv, D)
    vc = v.reshape(B, h_kv, nb, bs, D).transpose(0, 2, 3, 1, 4).reshape(B * nb, bs, h_kv, D)
    table = np.arange(B * nb).reshape(B, nb)
    o, lse = paged.paged_attn_fwd_ref(q, kc, vc, table, np.full(B, n_k), causal, 0.3)
    o_d, lse_d = orc.attn_fwd_ref(q, k, v, causal, 0.3)
    np.testing.assert_allclose(o, o_d, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, lse_d, rtol=1e-13, atol=1e-14)


def test_physical_block_placement_does_not_matter():
    rng = np.random.default_rng(4)
    kc, vc = rand_cache(12, 8, 2, 4, 5)
    table = np.array([[3, 7, 1, 9], [0, 11, 4, 2]])
    lens = np.array([29, 17])
    q = rng.standard_normal((2, 4, 2, 4))
    o, lse = paged.paged_attn_fwd_ref(q, kc, vc, table, lens, True, 0.5)
    perm = rng.permutation(12)           # physical block i moves to perm[i]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    o2, lse2 = paged.paged_attn_fwd_ref(q, kc2, vc2, perm[table], lens, True, 0.5)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_slots_past_the_context_are_ignored():
    # The last block's invalid tokens (and unused blocks) may hold anything.
    rng = np.random.default_rng(6)
    kc, vc = rand_cache(6, 8, 1, 4, 7)
    table = np.array([[4, 1, 5]])
    lens = np.array([13])                # block 1 holds 5 valid tokens of 8
    q = rng.standard_normal((1, 2, 3, 4))
    o, _ = paged.paged_attn_fwd_ref(q, kc, vc, table, lens, False, 0.5)
    kc[1, 5:] = 1e30
    vc[1, 5:] = np.nan
    kc[5] = -1e30
    vc[5] = np.inf
    o2, _ = paged.paged_attn_fwd_ref(q, kc, vc, table, lens, False, 0.5)
    np.testing.assert_array_equal(o, o2)


def test_reshape_and_cache_rule():
    rng = np.random.default_rng(8)
    kc = np.zeros((4, 8, 2, 3))
    vc = np.zeros((4, 8, 2, 3))
    k_new = rng.standard_normal((5, 2, 3))
    v_new = rng.standard_normal((5, 2, 3))
    slots = np.array([0, 17, -1, 31, 9])   # token 2 is skipped
    paged.reshape_and_cache(k_new, v_new, slots, kc, vc)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        np.testing.assert_array_equal(kc[s // 8, s % 8], k_new[i])
        np.testing.assert_array_equal(vc[s // 8, s % 8], v_new[i])
    assert np.count_nonzero(kc.any(axis=(2, 3))) == 4   # exactly the four written slots


def test_pins_catch_planted_paging_mistakes():
    rng = np.random.default_rng(9)
    kc, vc = rand_cache(8, 4, 1, 3, 10)
    table = np.array([[6, 2, 5]])
    lens = np.array([10])
    q = rng.standard_normal((1, 1, 2, 3))
    want = brute_paged(q, kc, vc, table, lens, True, float(np.float32(0.6)))
    # (a) using the logical block index as the physical one
    o_bad, _ = paged.paged_attn_fwd_ref(q, kc, vc, np.array([[0, 1, 2]]), lens, True, 0.6)
    assert not np.allclose(o_bad, want)
    # (b) offset taken from the wrong end of the block
    k_b = np.stack([kc[table[0][p // 4], 3 - p % 4] for p in range(10)], axis=1)[None]
    v_b = np.stack([vc[table[0][p // 4], 3 - p % 4] for p in range(10)], axis=1)[None]
    o_bad2, _ = orc.attn_fwd_ref(q, k_b, v_b, True, 0.6)
    assert not np.allclose(o_bad2, want)
    # (c) the whole last block attended to (no invalid-token mask)
    o_bad3, _ = paged.paged_attn_fwd_ref(q, kc, vc, table, np.array([12]), True, 0.6)
    assert not np.allclose(o_bad3, want)


# ---------------------------------------------------------- selected blocks


def full_selection(table, lens, h_kv, bs):
    """Every block of every sequence, in order, for every K/V head."""
    B = table.shape[0]
    nb = [(int(n) + bs - 1) // bs for n in lens]
    m = max(nb)
    pages = np.zeros((B, h_kv, m), dtype=np.int64)
    blocks = np.zeros((B, h_kv, m), dtype=np.int64)
    count = np.zeros((B, h_kv), dtype=np.int64)
    for b in range(B):
        for kvh in range(h_kv):
            pages[b, kvh, :nb[b]] = table[b, :nb[b]]
            blocks[b, kvh, :nb[b]] = np.arange(nb[b])
            count[b, kvh] = nb[b]
    return pages, blocks, count


@pytest.mark.parametrize("causal", [False, True])
def test_sparse_with_every_block_equals_paged(causal):
    rng = np.random.default_rng(20)
    kc, vc = rand_cache(10, 8, 2, 4, 21)
    table = np.array([[3, 7, 1, 9], [0, 2, 4, 6]])
    lens = np.array([29, 20])
    q = rng.standard_normal((2, 4, 3, 4))
    o, lse = paged.paged_attn_fwd_ref(q, kc, vc, table, lens, causal, 0.5)
    o2, lse2 = paged.sparse_attn_fwd_ref(q, kc, vc, *full_selection(table, lens, 2, 8), lens, causal, 0.5)
    np.testing.assert_allclose(o2, o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13, atol=1e-14)


def brute_sparse(q, kc, vc, pages, blocks, count, lens, causal, scale):
    B, H, n_q, D = q.shape
    bs, h_kv = kc.shape[1], kc.shape[2]
    o = np.zeros(q.shape)
    lse = np.full((B, H, n_q), -np.inf)
    for b in range(B):
        for h in range(H):
            kvh = h // (H // h_kv)
            for i in range(n_q):
                s = []
                for e in range(int(count[b, kvh])):
                    for r in range(bs):
                        p = int(blocks[b, kvh, e]) * bs + r
                        if p >= lens[b] or (causal and p > i + int(lens[b]) - n_q):
                            continue
                        pg = int(pages[b, kvh, e])
                        s.append((pg, r, scale * sum(q[b, h, i, t] * kc[pg, r, kvh, t] for t in range(D))))
                if not s:
                    continue
                mx = max(x for _, _, x in s)
                w = [(pg, r, math.exp(x - mx)) for pg, r, x in s]
                tot = sum(x for _, _, x in w)
                lse[b, h, i] = mx + math.log(tot)
                for t in range(D):
                    o[b, h, i, t] = sum(x * vc[pg, r, kvh, t] for pg, r, x in w) / tot
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_sparse_brute_force(causal):
    rng = np.random.default_rng(22)
    kc, vc = rand_cache(9, 4, 2, 3, 23)
    # per (sequence, K/V head): a few blocks of the context, out of order,
    # one of them wholly past the context (sequence 1: 9 tokens = blocks 0-2)
    pages = np.array([[[5, 1, 8], [2, 0, 0]], [[7, 3, 4], [6, 2, 0]]])
    blocks = np.array([[[2, 0, 4], [1, 0, 0]], [[1, 3, 0], [2, 0, 0]]])
    count = np.array([[3, 1], [3, 2]])
    lens = np.array([19, 9])
    q = rng.standard_normal((2, 4, 2, 3))
    sc = float(np.float32(0.8))
    o, lse = paged.sparse_attn_fwd_ref(q, kc, vc, pages, blocks, count, lens, causal, sc)
    bo, blse = brute_sparse(q, kc, vc, pages, blocks, count, lens, causal, sc)
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, blse, rtol=1e-12, atol=1e-13)


def test_sparse_selection_order_and_empty_rows():
    rng = np.random.default_rng(24)
    kc, vc = rand_cache(6, 8, 1, 4, 25)
    q = rng.standard_normal((1, 2, 1, 4))
    pages = np.array([[[4, 0, 5, 2]]])
    blocks = np.array([[[3, 0, 1, 2]]])
    lens = np.array([30])
    o, lse = paged.sparse_attn_fwd_ref(q, kc, vc, pages, blocks, np.array([[4]]), lens, False, 0.5)
    perm = [2, 0, 3, 1]
    o2, lse2 = paged.sparse_attn_fwd_ref(q, kc, vc, pages[:, :, perm], blocks[:, :, perm], np.array([[4]]), lens,
                                         False, 0.5)
    np.testing.assert_allclose(o2, o, rtol=1e-13, atol=1e-14)   # softmax over a set: order is irrelevant
    np.testing.assert_allclose(lse2, lse, rtol=1e-13, atol=1e-14)
    # only a block wholly past the context, or nothing selected: empty rows
    for cnt, blk in ((1, np.array([[[4, 0, 0, 0]]])), (0, blocks)):
        o3, lse3 = paged.sparse_attn_fwd_ref(q, kc, vc, pages, blk, np.array([[cnt]]), lens, False, 0.5)
        assert np.all(o3 == 0) and np.all(np.isneginf(lse3))


def test_pins_catch_planted_sparse_mistakes():
    rng = np.random.default_rng(26)
    kc, vc = rand_cache(8, 4, 1, 3, 27)
    q = rng.standard_normal((1, 1, 2, 3))
    pages = np.array([[[6, 1, 3]]])
    blocks = np.array([[[2, 0, 1]]])
    count = np.array([[3]])
    lens = np.array([10])                 # block 2 holds 2 valid tokens
    sc = float(np.float32(0.6))
    want, _ = brute_sparse(q, kc, vc, pages, blocks, count, lens, True, sc)
    # (a) positions from the entry index instead of the logical block
    bad, _ = paged.sparse_attn_fwd_ref(q, kc, vc, pages, np.array([[[0, 1, 2]]]), count, lens, True, sc)
    assert not np.allclose(bad, want)
    # (b) physical page taken as the logical block
    bad2, _ = paged.sparse_attn_fwd_ref(q, kc, vc, pages, pages, count, lens, True, sc)
    assert not np.allclose(bad2, want)


def merge_slices(parts):
    """Merge per-slice (O_s normalised by its own row sum, lse_s) results
    with the online-softmax rule: lse = log sum exp lse_s and O = sum
    exp(lse_s - lse) O_s; a slice with lse_s = -inf has weight 0."""
    lses = np.stack([l for _, l in parts])                      # [slices, rows]
    mx = np.max(lses, axis=0)
    lse = mx + np.log(np.sum(np.exp(lses - mx), axis=0))
    o = sum(np.exp(l - lse)[:, None] * np.nan_to_num(o_s) for o_s, l in parts)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_key_slices_merge_to_the_full_attention(causal):
    # The identity the split paged forward relies on, checked with the
    # oracle's one-head forward: attention over slices of the keys, merged,
    # equals attention over all of them.  Causal rows see only keys up to
    # their position, so some rows see nothing of the later slices
    # (lse_s = -inf there).
    rng = np.random.default_rng(77)
    n_q, n_k, d = 40, 300, 32
    q, k, v = (rng.standard_normal(s) for s in ((n_q, d), (n_k, d), (n_k, d)))
    scale = 1 / math.sqrt(d)
    full_o, full_lse = orc.attn_fwd_head(q, k, v, causal, scale)
    off = n_k - n_q                                          # queries are the last n_q positions
    parts = []
    for lo, hi in ((0, 100), (100, 255), (255, 270), (270, 300)):
        o_s = np.zeros((n_q, d))
        l_s = np.full(n_q, -np.inf)
        for i in range(n_q):
            top = min(hi, i + off + 1) if causal else hi     # one past the last key row i sees here
            if top > lo:
                o_i, l_i = orc.attn_fwd_head(q[i:i + 1], k[lo:top], v[lo:top], False, scale)
                o_s[i], l_s[i] = o_i[0], l_i[0]
        parts.append((o_s, l_s))
    if causal:
        assert np.isinf(parts[3][1]).any()                   # rows at positions 260-269 see nothing of keys 270-299
    o, lse = merge_slices(parts)
    assert np.max(np.abs(o - full_o)) < 1e-12
    assert np.max(np.abs(lse - full_lse)) < 1e-12
