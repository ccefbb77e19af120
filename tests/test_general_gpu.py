"""Grouped K/V heads, ragged lengths and unequal query / key lengths: CUDA
path (through the C ABI's general entry points) against the fp64 oracle on
the same seeded draws.

Shapes cover: N = 1, lengths that end inside a 128-row tile (and inside a
64-key tile for D = 256), several tiles plus a ragged tail, Nq < Nk (causal
diagonal moved by Nk - Nq, including a single decode query), Nq > Nk
(non-causal), and K/V heads shared by 2, 3, 4 and 8 query heads.
"""

import math

import pytest
import torch

from attention_sm_flashattention_gb300 import _native, api
from attention_sm_flashattention_gb300.inputs import make_inputs
from oracle import attention as orc

from helpers import (GRAD_RTOL, GRAD_RTOL_BF16, LSE_ATOL, O_ATOL, O_ATOL_BF16, max_abs, rel_fro,
                     sample_heads)

pytestmark = pytest.mark.gpu

# (Z, H, Hkv, Nq, Nk, D)
RAGGED = [
    (1, 2, 2, 1, 1, 64),
    (1, 2, 2, 77, 77, 64),
    (1, 2, 2, 129, 129, 128),
    (2, 3, 3, 200, 200, 128),
    (1, 2, 2, 383, 383, 64),
]
UNEQUAL = [
    (1, 2, 2, 100, 300, 64),
    (1, 2, 2, 1, 1000, 128),
    (1, 2, 2, 128, 512, 128),
    (1, 3, 3, 257, 700, 64),
    (1, 2, 2, 300, 100, 128),   # more queries than keys: non-causal only
]
GROUPED = [
    # few queries per head: the query heads of a K/V head are packed into
    # one tile (rows cycle through the query positions)
    (2, 8, 2, 8, 300, 128),
    (1, 16, 2, 16, 16, 64),
    (2, 4, 1, 1, 500, 256),
    (3, 6, 2, 40, 77, 128),
    (2, 8, 2, 256, 256, 128),
    (1, 4, 1, 384, 384, 64),
    (1, 6, 3, 200, 333, 128),
    (1, 8, 8, 130, 260, 64),
    (2, 8, 1, 64, 640, 128),
]
D256_FWD = [
    (1, 2, 2, 100, 100, 256),
    (1, 4, 2, 256, 256, 256),
    (1, 2, 2, 70, 333, 256),
]
D256_BWD = [
    (1, 2, 2, 256, 256, 256),
    (2, 1, 1, 384, 384, 256),
    (1, 2, 2, 1, 1, 256),
    (1, 2, 2, 100, 100, 256),
    (1, 4, 2, 200, 333, 256),
    (1, 4, 1, 130, 130, 256),
    (1, 2, 2, 300, 70, 256),
]


def ident(s):
    return "z%dh%dkv%dq%dk%dd%d" % s


def run_and_check(shape, causal, dtype=torch.float16, backward=True, seed_base=9100):
    Z, H, Hkv, Nq, Nk, D = shape
    seed = seed_base + Z * 7 + H * 11 + Hkv * 13 + Nq + 3 * Nk + D + int(causal)
    q, k, v, do = make_inputs(Z, H, Nq, D, seed, dtype=dtype, Hkv=Hkv, Nk=Nk)
    scale = 1 / math.sqrt(D)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    if causal and Nq > Nk:
        # a query row would see no key: refused before anything is enqueued
        with pytest.raises(_native.FaError) as e:
            api.fwd(qd, kd, vd, causal=causal, scale=scale)
        assert e.value.code == _native.FA_ERR_UNSUPPORTED
        return
    o, lse = api.fwd(qd, kd, vd, causal=causal, scale=scale)
    grads = api.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale) if backward else None
    assert api.device_status() == 0
    o_tol = O_ATOL_BF16 if dtype == torch.bfloat16 else O_ATOL
    g_tol = GRAD_RTOL_BF16 if dtype == torch.bfloat16 else GRAD_RTOL
    o_ref, lse_ref = orc.attn_fwd_ref(q, k, v, causal, scale)
    assert max_abs(o, o_ref) <= o_tol
    assert max_abs(lse, lse_ref) <= LSE_ATOL
    if backward:
        for name, g, r in zip(("dq", "dk", "dv"), grads, orc.attn_bwd_ref(q, k, v, do, causal, scale)):
            assert tuple(g.shape) == r.shape
            if not r.any():
                # every row sees one key (Nk = 1): the softmax is constant, dQ
                # and dK vanish exactly, and the GPU value is the rounding
                # residue of dP - Delta; a relative error has no meaning here
                assert max_abs(g, r) <= O_ATOL, name
                continue
            err = rel_fro(g, r)
            assert err <= g_tol, (name, err)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", RAGGED, ids=ident)
def test_ragged_lengths(shape, causal):
    run_and_check(shape, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", UNEQUAL, ids=ident)
def test_unequal_lengths(shape, causal):
    run_and_check(shape, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", GROUPED, ids=ident)
def test_grouped_heads(shape, causal):
    run_and_check(shape, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 4, 2, 200, 333, 128), (1, 4, 1, 129, 129, 64)], ids=ident)
def test_grouped_ragged_bf16(shape, causal):
    run_and_check(shape, causal, dtype=torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", D256_FWD, ids=ident)
def test_d256_forward_general(shape, causal):
    run_and_check(shape, causal, backward=False)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", D256_BWD, ids=ident)
def test_d256_backward_general(shape, causal):
    run_and_check(shape, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_d256_backward_general_bf16(causal):
    run_and_check((1, 4, 2, 200, 333, 256), causal, dtype=torch.bfloat16)


def test_output_rows_past_the_end_are_untouched():
    # A ragged last tile must not write past its head's rows: outputs are
    # stored into larger buffers whose tail holds a sentinel.
    Z, H, Hkv, Nq, Nk, D = 1, 2, 1, 77, 130, 64
    q, k, v, do = (t.cuda() for t in make_inputs(Z, H, Nq, D, 3, Hkv=Hkv, Nk=Nk))
    sentinel = 1234.0
    o_buf = torch.full((Z * H * Nq * D + 4096,), sentinel, dtype=torch.float16, device="cuda")
    lse_buf = torch.full((Z * H * Nq + 1024,), sentinel, dtype=torch.float32, device="cuda")
    o = o_buf[: Z * H * Nq * D].view(Z, H, Nq, D)
    lse = lse_buf[: Z * H * Nq].view(Z, H, Nq)
    api.fwd(q, k, v, causal=True, out=(o, lse))
    dk_buf = torch.full((Z * Hkv * Nk * D + 4096,), sentinel, dtype=torch.float16, device="cuda")
    dq_buf = torch.full((Z * H * Nq * D + 4096,), sentinel, dtype=torch.float16, device="cuda")
    dv_buf = torch.full((Z * Hkv * Nk * D + 4096,), sentinel, dtype=torch.float16, device="cuda")
    dq = dq_buf[: Z * H * Nq * D].view(Z, H, Nq, D)
    dk = dk_buf[: Z * Hkv * Nk * D].view(Z, Hkv, Nk, D)
    dv = dv_buf[: Z * Hkv * Nk * D].view(Z, Hkv, Nk, D)
    api.bwd(q, k, v, o, do, lse, causal=True, out=(dq, dk, dv))
    assert api.device_status() == 0
    for buf, n in ((o_buf, o.numel()), (lse_buf, lse.numel()), (dq_buf, dq.numel()), (dk_buf, dk.numel()),
                   (dv_buf, dv.numel())):
        assert bool((buf[n:] == sentinel).all())
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(dq).all()) and bool(torch.isfinite(dk).all())


# Larger shapes launched as a user would launch them, checked on sampled
# heads: a grouped-head causal shape (8 query heads per K/V head) and a
# ragged length near the benchmark's.
LARGE = [
    ("gqa_z16h32kv4n1024d128c", (16, 32, 4, 1024, 1024, 128), True),
    ("ragged_z32h8n1000d128", (32, 8, 8, 1000, 1000, 128), False),
    ("prefill_z8h16kv2q512k2048d64c", (8, 16, 2, 512, 2048, 64), True),
    ("gqa_z8h16kv4n1000d256c", (8, 16, 4, 1000, 1000, 256), True),
]


@pytest.mark.parametrize("name,shape,causal", LARGE, ids=[x[0] for x in LARGE])
def test_large_general_shapes_sampled_heads(name, shape, causal):
    Z, H, Hkv, Nq, Nk, D = shape
    q, k, v, do = make_inputs(Z, H, Nq, D, 9900 + Nq + Nk + D, Hkv=Hkv, Nk=Nk)
    scale = 1 / math.sqrt(D)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = api.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = api.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    assert api.device_status() == 0
    g = H // Hkv
    heads = sample_heads(Z * H, 3)
    o_ref, lse_ref = orc.attn_fwd_ref(q, k, v, causal, scale, heads=heads)
    dq_ref, dk_ref, dv_ref = orc.attn_bwd_ref(q, k, v, do, causal, scale, heads=heads)
    kv_heads = orc.sampled_kv_heads(heads, g)
    of, lf, dqf = o.reshape(Z * H, Nq, D), lse.reshape(Z * H, Nq), dq.reshape(Z * H, Nq, D)
    dkf, dvf = dk.reshape(Z * Hkv, Nk, D), dv.reshape(Z * Hkv, Nk, D)
    for i, h in enumerate(heads):
        assert max_abs(of[h], o_ref[i]) <= O_ATOL, (name, h)
        assert max_abs(lf[h], lse_ref[i]) <= LSE_ATOL, (name, h)
        assert rel_fro(dqf[h], dq_ref[i]) <= GRAD_RTOL, (name, "dq", h)
    for i, kvh in enumerate(kv_heads):
        assert rel_fro(dkf[kvh], dk_ref[i]) <= GRAD_RTOL, (name, "dk", kvh)
        assert rel_fro(dvf[kvh], dv_ref[i]) <= GRAD_RTOL, (name, "dv", kvh)


@pytest.mark.parametrize("causal", [False, True])
def test_d256_backward_inputs_only_16_byte_aligned(causal):
    # V and dO are read row by row by the D = 256 backward; views that start
    # 16 bytes into an allocation are 16- but not 32-byte aligned.
    Z, H, Hkv, Nq, Nk, D = 1, 4, 2, 200, 333, 256
    q, k, v, do = make_inputs(Z, H, Nq, D, 9700 + int(causal), Hkv=Hkv, Nk=Nk)
    scale = 1 / math.sqrt(D)

    def shifted(t):
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device="cuda")
        view = buf[8:].view(t.shape)
        view.copy_(t.cuda())
        assert view.data_ptr() % 32 == 16
        return view

    qd, kd = q.cuda(), k.cuda()
    vd, dod = shifted(v), shifted(do)
    o, lse = api.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = api.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    assert api.device_status() == 0
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), orc.attn_bwd_ref(q, k, v, do, causal, scale)):
        assert rel_fro(g, r) <= GRAD_RTOL, name
