"""Forward over selected blocks of a paged cache: CUDA path (fa_fwd_sparse
through the C ABI) against the fp64 oracle on the same seeded draws.

Selections are random subsets of each sequence's blocks per K/V head, in
shuffled order, including the block that holds the end of the context, a
block wholly past the context, and empty selections (rows with no visible
key: O = 0, lse = -inf).
"""

import math

import numpy as np
import pytest
import torch

from attention_sm_flashattention_gb300 import api
from attention_sm_flashattention_gb300.inputs import make_paged_inputs
from oracle import paged as porc

from helpers import LSE_ATOL, O_ATOL, O_ATOL_BF16, max_abs

pytestmark = pytest.mark.gpu


def make_selection(table, lens, h_kv, ps, keep, seed, extra_past=False, empty=()):
    """Per (sequence, K/V head): a random `keep` share of the context's
    blocks, shuffled; optionally one block wholly past the context; the
    (b, kvh) pairs in `empty` select nothing."""
    rng = np.random.default_rng(seed)
    B = table.shape[0]
    rows = []
    for b in range(B):
        nb = (int(lens[b]) + ps - 1) // ps
        for kvh in range(h_kv):
            if (b, kvh) in empty:
                rows.append(([], []))
                continue
            blocks = [int(x) for x in rng.permutation(nb)[:max(1, int(round(keep * nb)))]]
            if nb - 1 not in blocks:
                blocks.append(nb - 1)        # the block that holds the context's end
            rng.shuffle(blocks)
            pages = [int(table[b, x]) for x in blocks]
            if extra_past and nb < table.shape[1]:
                blocks.append(nb)            # logical block past the context: must contribute nothing
                pages.append(int(table[b, 0]))
            rows.append((pages, blocks))
    m = max(1, max(len(p) for p, _ in rows))
    sel_pages = np.zeros((B, h_kv, m), dtype=np.int32)
    sel_blocks = np.zeros((B, h_kv, m), dtype=np.int32)
    count = np.zeros((B, h_kv), dtype=np.int32)
    for idx, (p, bl) in enumerate(rows):
        b, kvh = divmod(idx, h_kv)
        sel_pages[b, kvh, :len(p)] = p
        sel_blocks[b, kvh, :len(bl)] = bl
        count[b, kvh] = len(p)
    return sel_pages, sel_blocks, count


# (B, H, Hkv, Nq, context_lens, D, page_size, keep)
CASES = [
    (3, 8, 2, 1, (77, 300, 1000), 128, 16, 0.5),
    (2, 4, 4, 1, (129, 2000), 64, 64, 0.3),
    (2, 8, 1, 1, (640, 65), 128, 128, 0.6),
    (2, 4, 2, 1, (200, 333), 256, 32, 0.5),
    (2, 6, 3, 64, (300, 713), 128, 32, 0.7),
    (1, 4, 2, 130, (500,), 256, 64, 0.5),
    (2, 8, 2, 4, (300, 700), 128, 64, 0.5),   # packed query heads
]


def ident(c):
    B, H, Hkv, Nq, lens, D, ps, keep = c
    return f"b{B}h{H}kv{Hkv}q{Nq}d{D}p{ps}k{keep}_" + "-".join(map(str, lens))


def run_case(case, causal, dtype=torch.float16, extra_past=False, empty=()):
    B, H, Hkv, Nq, lens, D, ps, keep = case
    seed = 8300 + B + 3 * H + Hkv + Nq + sum(lens) + D + ps + int(causal)
    q, kc, vc, table, cl = make_paged_inputs(B, H, Hkv, Nq, lens, D, ps, seed, dtype=dtype, spare_pages=4)
    sp, sb, cnt = make_selection(table.numpy(), lens, Hkv, ps, keep, seed, extra_past, empty)
    scale = 1 / math.sqrt(D)
    o, lse = api.fwd_sparse(q.cuda(), kc.cuda(), vc.cuda(), torch.from_numpy(sp).cuda(), torch.from_numpy(sb).cuda(),
                            torch.from_numpy(cnt).cuda(), cl.cuda(), causal=causal, scale=scale)
    assert api.device_status() == 0
    o_ref, lse_ref = porc.sparse_attn_fwd_ref(q, kc, vc, sp, sb, cnt, cl.numpy(), causal, scale)
    assert bool(torch.isfinite(o).all())
    tol = O_ATOL_BF16 if dtype == torch.bfloat16 else O_ATOL
    assert max_abs(o, o_ref) <= tol
    fin = np.isfinite(lse_ref)
    lse_h = lse.cpu().numpy()
    assert np.array_equal(np.isfinite(lse_h), fin)          # the same rows are empty
    if fin.any():
        assert float(np.max(np.abs(lse_h[fin] - lse_ref[fin]))) <= LSE_ATOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=ident)
def test_sparse_forward(case, causal):
    run_case(case, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_sparse_forward_block_past_context_and_empty_selection(causal):
    run_case(CASES[0], causal, extra_past=True, empty={(0, 1), (2, 0)})


def test_sparse_forward_bf16():
    run_case(CASES[4], True, dtype=torch.bfloat16)


def test_sparse_every_block_in_order_equals_paged():
    B, H, Hkv, Nq, D, ps = 2, 8, 2, 1, 128, 32
    lens = (300, 517)
    q, kc, vc, table, cl = (t.cuda() for t in make_paged_inputs(B, H, Hkv, Nq, lens, D, ps, 31))
    nb = table.shape[1]
    tab = table.cpu().numpy()
    sp = np.zeros((B, Hkv, nb), dtype=np.int32)
    sb = np.zeros((B, Hkv, nb), dtype=np.int32)
    cnt = np.zeros((B, Hkv), dtype=np.int32)
    for b in range(B):
        n = (lens[b] + ps - 1) // ps
        for kvh in range(Hkv):
            sp[b, kvh, :n] = tab[b, :n]
            sb[b, kvh, :n] = np.arange(n)
            cnt[b, kvh] = n
    o_s, lse_s = api.fwd_sparse(q, kc, vc, torch.from_numpy(sp).cuda(), torch.from_numpy(sb).cuda(),
                                torch.from_numpy(cnt).cuda(), cl, causal=True)
    o_p, lse_p = api.fwd_paged(q, kc, vc, table, cl, causal=True)
    assert api.device_status() == 0
    assert torch.equal(o_s, o_p)
    assert torch.equal(lse_s, lse_p)
