"""Paged forward with split key ranges: CUDA path (fa_fwd_paged_split through
the C ABI: the paged kernel over (work item, slice) units, then the merge
kernel) against the fp64 paged oracle on the same seeded draws.

Covers decode and chunked prefill, grouped heads (packed and not), every
head dimension, slice counts that do not divide the key tiles, more slices
than a short context has tiles (empty slices), causal rows that see no key
of a slice, bf16, and the library's own slice count.
"""

import math

import pytest
import torch

from attention_sm_flashattention_gb300 import _native, api
from attention_sm_flashattention_gb300.inputs import make_paged_inputs
from oracle import paged as porc

from helpers import LSE_ATOL, O_ATOL, O_ATOL_BF16, max_abs

pytestmark = pytest.mark.gpu

# (B, H, Hkv, Nq, context_lens, D, page_size, splits)
CASES = [
    (2, 8, 2, 1, (77, 3000), 128, 64, 4),
    (2, 8, 2, 1, (1000, 2999), 128, 32, 7),       # 7 slices of 8 and 24 key tiles
    (3, 4, 4, 1, (1, 40, 129), 64, 16, 6),          # more slices than tiles: empty slices
    (2, 4, 2, 1, (500, 1300), 256, 64, 5),
    (2, 8, 2, 16, (300, 700), 128, 32, 5),          # packed, causal positions cycle every 16 rows
    (1, 4, 2, 130, (900,), 128, 64, 3),             # two query tiles, paired in one causal unit
    (1, 4, 2, 128, (301,), 128, 64, 3),             # causal: rows at positions 173-255 see nothing of slice 2
    (2, 12, 3, 5, (37, 260), 64, 16, 3),
]


def ident(c):
    B, H, Hkv, Nq, lens, D, ps, sp = c
    return f"b{B}h{H}kv{Hkv}q{Nq}d{D}p{ps}s{sp}_" + "-".join(map(str, lens))


def poison_unreadable(kc, vc, table, lens, ps):
    """Inf / NaN in every cache slot no sequence may read: past each context
    in its last page, and the spare pages."""
    used = set()
    for b, n in enumerate(lens):
        pages = table[b, :(n + ps - 1) // ps].tolist()
        used.update(pages)
        if n % ps:
            kc[pages[-1], n % ps:] = float("inf")
            vc[pages[-1], n % ps:] = float("nan")
    for pg in range(kc.shape[0]):
        if pg not in used:
            kc[pg] = float("nan")
            vc[pg] = float("inf")


def run_case(case, causal, dtype=torch.float16, splits=None, poison=False):
    B, H, Hkv, Nq, lens, D, ps, sp = case
    if splits is not None:
        sp = splits
    seed = 9100 + B + 3 * H + Hkv + Nq + sum(lens) + D + ps + int(causal)
    q, kc, vc, table, cl = make_paged_inputs(B, H, Hkv, Nq, lens, D, ps, seed, dtype=dtype)
    if poison:
        poison_unreadable(kc, vc, table, lens, ps)
    scale = 1 / math.sqrt(D)
    o, lse = api.fwd_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cl.cuda(), causal=causal, scale=scale,
                           splits=sp)
    assert api.device_status() == 0
    o_ref, lse_ref = porc.paged_attn_fwd_ref(q, kc, vc, table.numpy(), cl.numpy(), causal, scale)
    assert bool(torch.isfinite(o).all())
    tol = O_ATOL_BF16 if dtype == torch.bfloat16 else O_ATOL
    assert max_abs(o, o_ref) <= tol
    assert max_abs(lse, lse_ref) <= LSE_ATOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=ident)
def test_paged_split_forward(case, causal):
    run_case(case, causal)


def test_paged_split_forward_bf16():
    run_case(CASES[1], True, dtype=torch.bfloat16)


def test_paged_split_forward_bf16_d256():
    run_case(CASES[3], False, dtype=torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[3], CASES[6]], ids=ident)
def test_paged_split_forward_ignores_unreadable_slots(case, causal):
    run_case(case, causal, poison=True)


def test_paged_split_library_count():
    # splits=0: the library's count for this small batch (more than one on a
    # GPU with more SMs than work items)
    B, H, Hkv, Nq, lens, D, ps, _ = CASES[1]
    n = api.paged_split_count(B, H, Hkv, Nq, D, ps, 3000 // ps + 1, True)
    assert n > 1
    run_case(CASES[1], True, splits=0)


def test_paged_split_one_slice_is_the_paged_call():
    B, H, Hkv, Nq, lens, D, ps, _ = CASES[0]
    q, kc, vc, table, cl = (t.cuda() for t in make_paged_inputs(B, H, Hkv, Nq, lens, D, ps, 77))
    o1, l1 = api.fwd_paged(q, kc, vc, table, cl, causal=True, splits=1)
    o0, l0 = api.fwd_paged(q, kc, vc, table, cl, causal=True)
    assert api.device_status() == 0
    assert torch.equal(o1, o0) and torch.equal(l1, l0)


def test_paged_split_rejects_a_short_workspace():
    B, H, Hkv, Nq, lens, D, ps, sp = CASES[0]
    q, kc, vc, table, cl = (t.cuda() for t in make_paged_inputs(B, H, Hkv, Nq, lens, D, ps, 78))
    need = _native.lib().fa_fwd_paged_split_workspace_size(B, H, Nq, D, sp)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(_native.FaError) as e:
        api.fwd_paged(q, kc, vc, table, cl, splits=sp, workspace=ws)
    assert e.value.code == _native.FA_ERR_WORKSPACE


# A small decode batch with long contexts, the case splitting is for: 4
# sequences, 32 query heads over 8 K/V heads, contexts of 4k-32k tokens in
# 64-token pages; checked on sampled sequences.
def test_paged_split_small_batch_long_context_sampled():
    B, H, Hkv, D, ps = 4, 32, 8, 128, 64
    lens = [32768, 4097, 20000, 31111]
    q, kc, vc, table, cl = make_paged_inputs(B, H, Hkv, 1, lens, D, ps, 13, spare_pages=1)
    o, lse = api.fwd_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cl.cuda(), causal=True, splits=0)
    assert api.device_status() == 0
    for b in (0, 1):
        o_ref, lse_ref = porc.paged_attn_fwd_ref(q[b:b + 1], kc, vc, table[b:b + 1].numpy(), cl[b:b + 1].numpy(),
                                                 True, 1 / math.sqrt(D))
        assert max_abs(o[b:b + 1], o_ref) <= O_ATOL, b
        assert max_abs(lse[b:b + 1], lse_ref) <= LSE_ATOL, b
