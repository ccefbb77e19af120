"""Forward over a paged K/V cache: CUDA path (fa_fwd_paged through the C ABI)
against the fp64 paged oracle on the same seeded draws.

Covers decode (one query per sequence) and chunked prefill (many queries at
the end of a longer context), grouped heads, every supported page size,
context lengths that end inside a page and inside a key tile, block-table
entries past a sequence's pages (set to -1), and NaN / Inf in cache slots
that no sequence may read.
"""

import math

import numpy as np
import pytest
import torch

from attention_sm_flashattention_gb300 import _native, api
from attention_sm_flashattention_gb300.inputs import make_paged_inputs
from oracle import attention as orc
from oracle import paged as porc

from helpers import LSE_ATOL, O_ATOL, O_ATOL_BF16, max_abs

pytestmark = pytest.mark.gpu

# (B, H, Hkv, Nq, context_lens, D, page_size)
CASES = [
    (3, 8, 2, 1, (1, 77, 300), 128, 16),
    (2, 4, 4, 1, (129, 1000), 64, 32),
    (2, 8, 1, 1, (640, 65), 128, 64),
    (2, 4, 2, 1, (256, 130), 128, 128),
    (2, 4, 2, 1, (200, 63), 256, 64),
    (2, 4, 2, 1, (33, 100), 256, 16),
    (2, 6, 3, 200, (300, 713), 128, 32),
    (1, 4, 2, 128, (128,), 64, 16),
    (2, 4, 4, 130, (500, 131), 256, 32),
    (2, 8, 2, 16, (300, 500), 128, 32),     # packed query heads, causal positions cycle every 16 rows
    (2, 12, 3, 5, (37, 260), 64, 16),
]


def ident(c):
    B, H, Hkv, Nq, lens, D, ps = c
    return f"b{B}h{H}kv{Hkv}q{Nq}d{D}p{ps}_" + "-".join(map(str, lens))


def run_case(case, causal, dtype=torch.float16, poison=False):
    B, H, Hkv, Nq, lens, D, ps = case
    seed = 7100 + B + 3 * H + Hkv + Nq + sum(lens) + D + ps + int(causal)
    q, kc, vc, table, cl = make_paged_inputs(B, H, Hkv, Nq, lens, D, ps, seed, dtype=dtype)
    if poison:
        # slots no sequence may read: past each context in its last page, and
        # the spare pages
        used = set()
        for b in range(B):
            n = lens[b]
            pages = table[b, :(n + ps - 1) // ps].tolist()
            used.update(pages)
            if n % ps:
                kc[pages[-1], n % ps:] = float("inf")
                vc[pages[-1], n % ps:] = float("nan")
        for pg in range(kc.shape[0]):
            if pg not in used:
                kc[pg] = float("nan")
                vc[pg] = float("inf")
    scale = 1 / math.sqrt(D)
    o, lse = api.fwd_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cl.cuda(), causal=causal, scale=scale)
    assert api.device_status() == 0
    o_ref, lse_ref = porc.paged_attn_fwd_ref(q, kc, vc, table.numpy(), cl.numpy(), causal, scale)
    assert bool(torch.isfinite(o).all())
    tol = O_ATOL_BF16 if dtype == torch.bfloat16 else O_ATOL
    assert max_abs(o, o_ref) <= tol
    assert max_abs(lse, lse_ref) <= LSE_ATOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=ident)
def test_paged_forward(case, causal):
    run_case(case, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", [CASES[0], CASES[4], CASES[6]], ids=ident)
def test_paged_forward_ignores_unreadable_slots(case, causal):
    run_case(case, causal, poison=True)


@pytest.mark.parametrize("case", [CASES[1], CASES[6]], ids=ident)
def test_paged_forward_bf16(case):
    run_case(case, True, dtype=torch.bfloat16)


def test_paged_forward_matches_dense_call_on_contiguous_pages():
    # The same keys laid out page by page in order: the paged call and the
    # dense fa_fwd_ex call run the same arithmetic on the same tiles.
    B, H, Hkv, N, D, ps = 2, 8, 2, 384, 128, 64
    g = torch.Generator().manual_seed(5)
    q = torch.randn((B, H, N, D), generator=g).half().cuda()
    k = torch.randn((B, Hkv, N, D), generator=g).half().cuda()
    v = torch.randn((B, Hkv, N, D), generator=g).half().cuda()
    npg = N // ps
    kc = k.view(B, Hkv, npg, ps, D).permute(0, 2, 3, 1, 4).reshape(B * npg, ps, Hkv, D).contiguous()
    vc = v.view(B, Hkv, npg, ps, D).permute(0, 2, 3, 1, 4).reshape(B * npg, ps, Hkv, D).contiguous()
    table = torch.arange(B * npg, dtype=torch.int32, device="cuda").view(B, npg)
    cl = torch.full((B,), N, dtype=torch.int32, device="cuda")
    o_p, lse_p = api.fwd_paged(q, kc, vc, table, cl, causal=True)
    o_d, lse_d = api.fwd(q, k, v, causal=True)
    assert api.device_status() == 0
    assert torch.equal(o_p, o_d)
    assert torch.equal(lse_p, lse_d)


def test_paged_rejects_unsupported_page_sizes():
    q, kc, vc, table, cl = (t.cuda() for t in make_paged_inputs(1, 2, 2, 1, (40,), 256, 128, 1))
    with pytest.raises(_native.FaError) as e:
        api.fwd_paged(q, kc, vc, table, cl)          # D = 256 takes pages of at most 64 rows
    assert e.value.code == _native.FA_ERR_UNSUPPORTED


# A decode batch of the size a serving step would run, checked on sampled
# sequences: 64 sequences, 32 query heads over 8 K/V heads, contexts of
# 1-4096 tokens in 64-token pages.
def test_paged_decode_batch_sampled():
    B, H, Hkv, D, ps = 64, 32, 8, 128, 64
    lens = [int(x) for x in np.random.default_rng(11).integers(1, 4097, size=B)]
    q, kc, vc, table, cl = make_paged_inputs(B, H, Hkv, 1, lens, D, ps, 12)
    o, lse = api.fwd_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cl.cuda(), causal=True)
    assert api.device_status() == 0
    for b in (0, 17, 63):
        o_ref, lse_ref = porc.paged_attn_fwd_ref(q[b:b + 1], kc, vc, table[b:b + 1].numpy(), cl[b:b + 1].numpy(),
                                                 True, 1 / math.sqrt(D))
        assert max_abs(o[b:b + 1], o_ref) <= O_ATOL, b
        assert max_abs(lse[b:b + 1], lse_ref) <= LSE_ATOL, b


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("T,Hkv,D,num_pages,ps", [(37, 2, 64, 8, 16), (300, 8, 128, 12, 64), (5, 4, 256, 3, 32)])
def test_reshape_and_cache_matches_oracle(T, Hkv, D, num_pages, ps, dtype):
    g = torch.Generator().manual_seed(T + D)
    k_new = torch.randn((T, Hkv, D), generator=g).to(dtype)
    v_new = torch.randn((T, Hkv, D), generator=g).to(dtype)
    rows = num_pages * ps
    slots = torch.randperm(rows, generator=g)[:T].to(torch.int64)
    slots[::7] = -1                     # skipped tokens
    if T > 3:
        slots[3] = rows + 5             # outside the cache: skipped, never written
    kc = torch.randn((num_pages, ps, Hkv, D), generator=g).to(dtype)
    vc = torch.randn((num_pages, ps, Hkv, D), generator=g).to(dtype)
    kc_d, vc_d = kc.cuda(), vc.cuda()
    api.reshape_and_cache(k_new.cuda(), v_new.cuda(), slots.cuda(), kc_d, vc_d)
    torch.cuda.synchronize()
    kc_ref, vc_ref = kc.float().numpy().copy(), vc.float().numpy().copy()
    keep = slots < rows
    porc.reshape_and_cache(k_new.float().numpy()[keep.numpy()], v_new.float().numpy()[keep.numpy()],
                           slots.numpy()[keep.numpy()], kc_ref, vc_ref)
    # a pure copy: bit-exact
    assert np.array_equal(kc_d.float().cpu().numpy(), kc_ref)
    assert np.array_equal(vc_d.float().cpu().numpy(), vc_ref)


def test_cache_written_then_attended_equals_dense():
    # Decode-style round trip: write each sequence's tokens into scattered
    # pages with the cache write, then attend through the block table.
    B, H, Hkv, N, D, ps = 3, 8, 2, 200, 128, 32
    g = torch.Generator().manual_seed(21)
    k = torch.randn((B, Hkv, N, D), generator=g).half()
    v = torch.randn((B, Hkv, N, D), generator=g).half()
    q = torch.randn((B, H, 1, D), generator=g).half()
    npg = (N + ps - 1) // ps
    num_pages = B * npg + 2
    perm = torch.randperm(num_pages, generator=g)
    table = perm[:B * npg].view(B, npg).to(torch.int32)
    pos = torch.arange(N)
    slots = (table[:, pos // ps].to(torch.int64) * ps + (pos % ps)).reshape(-1)      # [B * N]
    kc = torch.zeros((num_pages, ps, Hkv, D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    api.reshape_and_cache(k.permute(0, 2, 1, 3).reshape(B * N, Hkv, D).contiguous().cuda(),
                          v.permute(0, 2, 1, 3).reshape(B * N, Hkv, D).contiguous().cuda(), slots.cuda(), kc, vc)
    cl = torch.full((B,), N, dtype=torch.int32, device="cuda")
    o, lse = api.fwd_paged(q.cuda(), kc, vc, table.cuda(), cl, causal=True)
    assert api.device_status() == 0
    o_ref, lse_ref = orc.attn_fwd_ref(q, k, v, True, 1 / math.sqrt(D))
    assert max_abs(o, o_ref) <= O_ATOL
    assert max_abs(lse, lse_ref) <= LSE_ATOL
