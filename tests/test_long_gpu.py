"""Long sequences: the forward at N = 16384 checked on sampled query rows,
the backward at N = 4096 checked in full, against the fp64 oracle.

A sampled row i of the forward is, by definition, attention of the single
query i over the keys it sees (0 .. i when causal, all of them otherwise),
which the oracle's one-head forward computes directly.
"""

import math

import pytest
import torch

from attention_sm_flashattention_gb300 import api
from attention_sm_flashattention_gb300.inputs import make_inputs
from oracle import attention as orc

from helpers import GRAD_RTOL, LSE_ATOL, O_ATOL, max_abs, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_forward_16k_sampled_rows(D, causal):
    Z, H, N = 1, 2, 16384
    q, k, v, _ = make_inputs(Z, H, N, D, seed=16000 + D + int(causal))
    scale = 1 / math.sqrt(D)
    o, lse = api.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    assert api.device_status() == 0
    o, lse = o.cpu(), lse.cpu()
    for h in range(H):
        for i in (0, 1, 127, 128, 4097, 8191, 12345, N - 1):
            n_keys = i + 1 if causal else N
            o_ref, lse_ref = orc.attn_fwd_head(q[0, h, i:i + 1], k[0, h, :n_keys], v[0, h, :n_keys], False, scale)
            assert max_abs(o[0, h, i:i + 1], o_ref) <= O_ATOL, (h, i)
            assert max_abs(lse[0, h, i:i + 1], lse_ref) <= LSE_ATOL, (h, i)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_4k(causal):
    Z, H, Hkv, N, D = 1, 2, 1, 4096, 128
    q, k, v, do = make_inputs(Z, H, N, D, seed=4096 + int(causal), Hkv=Hkv)
    scale = 1 / math.sqrt(D)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = api.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = api.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    assert api.device_status() == 0
    o_ref, lse_ref = orc.attn_fwd_ref(q, k, v, causal, scale)
    assert max_abs(o, o_ref) <= O_ATOL
    assert max_abs(lse, lse_ref) <= LSE_ATOL
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), orc.attn_bwd_ref(q, k, v, do, causal, scale)):
        assert rel_fro(got, ref) <= GRAD_RTOL, name
