"""bf16 forward and backward: CUDA path (through the C ABI) against the fp64
oracle on the same seeded draws rounded to bf16 instead of fp16."""

import math

import pytest
import torch

from attention_sm_flashattention_gb300 import _native, api
from attention_sm_flashattention_gb300.inputs import make_inputs
from oracle import attention as orc

from helpers import GRAD_RTOL_BF16, LSE_ATOL, O_ATOL_BF16, max_abs, rel_fro

pytestmark = pytest.mark.gpu

SMALL = [(1, 2, 128, 64), (2, 3, 384, 64), (1, 2, 256, 128), (2, 2, 512, 128), (1, 1, 128, 256), (1, 2, 384, 256)]


def bf16_inputs(Z, H, N, D, seed):
    return make_inputs(Z, H, N, D, seed=seed, dtype=torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "z%dh%dn%dd%d" % s)
def test_bf16_fwd_bwd_small_full_compare(shape, causal):
    Z, H, N, D = shape
    q, k, v, do = bf16_inputs(Z, H, N, D, seed=7000 + N + D + int(causal))
    scale = 1 / math.sqrt(D)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = api.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = api.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    assert api.device_status() == 0
    assert o.dtype == torch.bfloat16 and dq.dtype == torch.bfloat16
    o_ref, lse_ref = orc.attn_fwd_ref(q, k, v, causal, scale)
    assert max_abs(o, o_ref) <= O_ATOL_BF16
    assert max_abs(lse, lse_ref) <= LSE_ATOL
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), orc.attn_bwd_ref(q, k, v, do, causal, scale)):
        err = rel_fro(g, r)
        assert err <= GRAD_RTOL_BF16, (name, err)


def test_bf16_rejects_mixed_dtypes():
    q, k, v, _ = bf16_inputs(1, 1, 128, 64, seed=1)
    with pytest.raises(ValueError):
        api.fwd(q.cuda(), k.cuda().half(), v.cuda())


def test_bf16_c_abi_shares_fp16_error_codes():
    lib = _native.lib()
    rc = lib.fa_fwd_bf16(None, None, None, None, None, 1, 1, 128, 64, 0, 0.125, None)
    assert rc == _native.FA_ERR_INVALID_ARG
