"""Run-to-run determinism: every output tile has one writer and no kernel
accumulates across CTAs, so identical calls on identical inputs give
identical bits.  A race between warps (a buffer reused before its reader
finished, a barrier phase skipped) shows up here as a difference between
repeated calls, at sizes with several waves of the persistent grid."""

import pytest
import torch

from attention_sm_flashattention_gb300 import api
from attention_sm_flashattention_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

SHAPES = [(16, 8, 1024, 64), (16, 8, 1024, 128), (8, 8, 1024, 256), (4, 8, 1000, 128)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "z%dh%dn%dd%d" % s)
def test_repeated_calls_give_identical_bits(shape, causal):
    Z, H, N, D = shape
    q, k, v, do = (t.cuda() for t in make_inputs(Z, H, N, D, seed=4000 + D + int(causal)))
    first = None
    for _ in range(3):
        o, lse = api.fwd(q, k, v, causal=causal)
        dq, dk, dv = api.bwd(q, k, v, o, do, lse, causal=causal)
        torch.cuda.synchronize()
        assert api.device_status() == 0
        outs = (o, lse, dq, dk, dv)
        if first is None:
            first = tuple(t.clone() for t in outs)
            continue
        for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), first, outs):
            assert torch.equal(a, b), f"{name} differs between identical calls"
