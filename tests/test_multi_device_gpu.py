"""Two devices in one process: the kernels' function attributes (the raised
dynamic shared-memory limit) are set per device, so a call on a second GPU
after one on the first runs and matches the oracle.  Skipped when fewer than
two GPUs are visible."""

import math

import pytest
import torch

from attention_sm_flashattention_gb300 import api
from attention_sm_flashattention_gb300.inputs import make_inputs
from oracle import attention as orc

from helpers import GRAD_RTOL, LSE_ATOL, O_ATOL, max_abs, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.skipif(not torch.cuda.is_available() or torch.cuda.device_count() < 2,
                    reason="needs two visible GPUs")
@pytest.mark.parametrize("D", [64, 128, 256])
def test_fwd_bwd_on_second_device_after_first(D):
    Z, H, N, causal = 1, 2, 256, True
    q, k, v, do = make_inputs(Z, H, N, D, seed=77 + D)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = orc.attn_fwd_ref(q, k, v, causal, scale)
    dq_ref, dk_ref, dv_ref = orc.attn_bwd_ref(q, k, v, do, causal, scale)
    for dev in (0, 1):
        with torch.cuda.device(dev):
            qd, kd, vd, dod = (t.cuda(dev) for t in (q, k, v, do))
            o, lse = api.fwd(qd, kd, vd, causal=causal, scale=scale)
            dq, dk, dv = api.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
            torch.cuda.synchronize(dev)
            assert api.device_status() == 0
            assert max_abs(o, o_ref) <= O_ATOL
            assert max_abs(lse, lse_ref) <= LSE_ATOL
            for g, ref in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
                assert rel_fro(g, ref) <= GRAD_RTOL
