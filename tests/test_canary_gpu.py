"""Out-of-bounds writes: every output of the CUDA path is a view into a
larger device buffer whose guard regions (before and after the view) hold
a canary pattern; after the call the guards must be bit-for-bit unchanged
and the outputs still match the oracle.

Shapes are ragged (the last query and key tiles are partial, where TMA
stores clip and masks apply), with grouped heads, the D = 256 kernels and
the split paged forward, whose fp32 partial rows are written from
registers.  This stands in for a memory-checking tool on this GPU pool.
"""

import math

import pytest
import torch

from attention_sm_flashattention_gb300 import _native, api
from attention_sm_flashattention_gb300.inputs import make_inputs, make_paged_inputs
from oracle import attention as orc
from oracle import paged as porc

from helpers import GRAD_RTOL, LSE_ATOL, O_ATOL, max_abs, rel_fro

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements on each side (keeps 16-byte alignment for every dtype)


class Guarded:
    """Device tensors of the given shapes, each carved out of a buffer with
    GUARD canary elements before and after it."""

    def __init__(self):
        self.bufs = []

    def make(self, shape, dtype):
        n = math.prod(shape)
        buf = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        # a fixed bit pattern, distinct from anything the kernels write
        buf.view(torch.int16 if buf.element_size() == 2 else torch.int32).fill_(0x5A5A if buf.element_size() == 2
                                                                               else 0x5A5A5A5A)
        self.bufs.append((buf, n))
        return buf[GUARD:GUARD + n].view(shape)

    def check(self):
        torch.cuda.synchronize()
        for buf, n in self.bufs:
            raw = buf.view(torch.int16 if buf.element_size() == 2 else torch.int32)
            want = 0x5A5A if buf.element_size() == 2 else 0x5A5A5A5A
            assert bool((raw[:GUARD] == want).all()), "write before the output"
            assert bool((raw[GUARD + n:] == want).all()), "write after the output"


# (Z, H, Hkv, Nq, Nk, D, causal)
CASES = [
    (2, 3, 3, 200, 200, 128, True),
    (2, 4, 2, 77, 333, 64, False),
    (1, 4, 1, 130, 260, 128, True),
    (2, 2, 2, 100, 100, 256, True),
    (1, 2, 2, 1, 65, 128, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "z{}h{}kv{}q{}k{}d{}{}".format(*c[:6], "c" if c[6] else ""))
def test_outputs_stay_inside_their_buffers(case):
    Z, H, Hkv, Nq, Nk, D, causal = case
    q, k, v, do = make_inputs(Z, H, Nq, D, seed=500 + Nq + Nk + D, Hkv=Hkv, Nk=Nk)
    scale = 1 / math.sqrt(D)
    g = Guarded()
    o = g.make((Z, H, Nq, D), torch.float16)
    lse = g.make((Z, H, Nq), torch.float32)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    api.fwd(qd, kd, vd, causal=causal, scale=scale, out=(o, lse))
    dq = g.make((Z, H, Nq, D), torch.float16)
    dk = g.make((Z, Hkv, Nk, D), torch.float16)
    dv = g.make((Z, Hkv, Nk, D), torch.float16)
    api.bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale, out=(dq, dk, dv))
    assert api.device_status() == 0
    g.check()
    o_ref, lse_ref = orc.attn_fwd_ref(q, k, v, causal, scale)
    assert max_abs(o, o_ref) <= O_ATOL
    assert max_abs(lse, lse_ref) <= LSE_ATOL
    dq_ref, dk_ref, dv_ref = orc.attn_bwd_ref(q, k, v, do, causal, scale)
    for got, ref in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        assert rel_fro(got, ref) <= GRAD_RTOL


@pytest.mark.parametrize("splits", [1, 3])
def test_paged_outputs_stay_inside_their_buffers(splits):
    B, H, Hkv, Nq, lens, D, ps = 2, 8, 2, 3, (150, 700), 128, 32
    q, kc, vc, table, cl = make_paged_inputs(B, H, Hkv, Nq, lens, D, ps, 612)
    g = Guarded()
    o = g.make((B, H, Nq, D), torch.float16)
    lse = g.make((B, H, Nq), torch.float32)
    ws = None
    if splits > 1:  # the per-slice partial results are guarded too
        need = _native.lib().fa_fwd_paged_split_workspace_size(B, H, Nq, D, splits)
        ws = g.make((need // 4,), torch.int32)
    api.fwd_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cl.cuda(), causal=True, out=(o, lse), splits=splits,
                  workspace=ws)
    assert api.device_status() == 0
    g.check()
    o_ref, lse_ref = porc.paged_attn_fwd_ref(q, kc, vc, table.numpy(), cl.numpy(), True, 1 / math.sqrt(D))
    assert max_abs(o, o_ref) <= O_ATOL
    assert max_abs(lse, lse_ref) <= LSE_ATOL
