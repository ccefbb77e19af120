"""Backward parity: CUDA path (through the C ABI) against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

from attention_sm_flashattention_gb300 import api
from attention_sm_flashattention_gb300.inputs import make_inputs
from oracle import attention as orc

from helpers import GRAD_RTOL, rel_fro

pytestmark = pytest.mark.gpu


def run(q, k, v, do, causal, scale):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = api.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = api.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    assert api.device_status() == 0
    return dq, dk, dv


SMALL = [
    (1, 2, 128, 64), (1, 1, 256, 64), (2, 3, 384, 64),
    (1, 1, 128, 128), (1, 2, 256, 128), (2, 2, 512, 128),
    (1, 1, 128, 256), (1, 2, 384, 256),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "z%dh%dn%dd%d" % s)
def test_bwd_small_full_compare(shape, causal):
    Z, H, N, D = shape
    q, k, v, do = make_inputs(Z, H, N, D, seed=Z * 1000 + H * 100 + N + D + int(causal) + 7)
    scale = 1 / math.sqrt(D)
    dq, dk, dv = run(q, k, v, do, causal, scale)
    ref = orc.attn_bwd_ref(q, k, v, do, causal, scale)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        err = rel_fro(g, r)
        assert err <= GRAD_RTOL, (name, err)


def test_bwd_from_oracle_forward():
    # The backward alone: O and lse taken from the oracle instead of fa_fwd.
    Z, H, N, D = 1, 2, 256, 128
    q, k, v, do = make_inputs(Z, H, N, D, seed=31)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = orc.attn_fwd_ref(q, k, v, True, scale)
    o = torch.from_numpy(o_ref).to(torch.float16).cuda()
    lse = torch.from_numpy(lse_ref).to(torch.float32).cuda()
    dq, dk, dv = api.bwd(q.cuda(), k.cuda(), v.cuda(), o, do.cuda(), lse, causal=True, scale=scale)
    assert api.device_status() == 0
    ref = orc.attn_bwd_ref(q, k, v, do, True, scale)
    for g, r in zip((dq, dk, dv), ref):
        assert rel_fro(g, r) <= GRAD_RTOL


@pytest.mark.parametrize("D", [64, 128, 256])
def test_bwd_gradient_sum_invariants(D):
    # Rows of P sum to one and rows of dS to zero: sum_j dV_j = sum_i dO_i and
    # sum_j dK_j = 0 (up to fp16 rounding of the outputs).
    q, k, v, do = make_inputs(1, 1, 256, D, seed=40 + D)
    dq, dk, dv = run(q, k, v, do, False, 1 / math.sqrt(D))
    sdv = dv.double().sum(dim=2).cpu().numpy()
    sdo = do.double().sum(dim=2).numpy()
    assert np.max(np.abs(sdv - sdo)) <= 2e-2 * max(1.0, np.max(np.abs(sdo)))
    sdk = dk.double().sum(dim=2).cpu().numpy()
    assert np.max(np.abs(sdk)) <= 2e-2 * max(1.0, float(dk.double().abs().sum(dim=2).max()))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_deterministic(causal):
    q, k, v, do = make_inputs(2, 4, 512, 128, seed=12)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = api.fwd(qd, kd, vd, causal=causal)
    a = api.bwd(qd, kd, vd, o, dod, lse, causal=causal)
    b = api.bwd(qd, kd, vd, o, dod, lse, causal=causal)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_workspace_is_reusable_and_checked():
    Z, H, N, D = 1, 2, 256, 64
    q, k, v, do = make_inputs(Z, H, N, D, seed=13)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = api.fwd(qd, kd, vd)
    need = api.bwd_workspace_size(Z, H, N, D, False)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")  # garbage on entry is fine
    g1 = api.bwd(qd, kd, vd, o, dod, lse, workspace=ws)
    g2 = api.bwd(qd, kd, vd, o, dod, lse, workspace=ws)
    for x, y in zip(g1, g2):
        assert torch.equal(x, y)
    with pytest.raises(RuntimeError):
        api.bwd(qd, kd, vd, o, dod, lse, workspace=ws[: need - 256])
