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
