"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot hand the backward a workspace: they run inside a memory
pool or arena they do not own, or at a point where allocation calls are not
allowed.  fa_bwd_noalloc takes no workspace and allocates nothing; its scratch
is a fixed buffer built into the library.  These tests call it through the C
ABI and check that two calls in a row each give what fa_bwd gives on the same
inputs, and that a problem too large for the buffer is refused up front.

This file is collected last on purpose, so that a failure here cannot stop a
``-x`` run before the other tests have run.
"""

import ctypes
import math

import pytest
import torch

from attention_sm_flashattention_gb300 import _native, api
from attention_sm_flashattention_gb300.inputs import make_inputs

from helpers import GRAD_RTOL, rel_fro

pytestmark = pytest.mark.gpu


def noalloc_bwd(q, k, v, o, do, lse, causal, scale):
    Z, H, N, D = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    stream = torch.cuda.current_stream().cuda_stream
    rc = _native.lib().fa_bwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), Z, H, N, D, int(causal), float(scale), stream)
    assert rc == _native.FA_OK, _native.error_string(rc)
    return dq, dk, dv


@pytest.mark.parametrize("shape,causal", [((2, 4, 512, 128), False), ((1, 3, 384, 64), True),
                                          ((1, 2, 256, 256), True)])
def test_noalloc_matches_workspace_backward_twice(shape, causal):
    Z, H, N, D = shape
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = (t.cuda() for t in make_inputs(Z, H, N, D, seed=500 + D))
    o, lse = api.fwd(q, k, v, causal=causal, scale=scale)
    want = api.bwd(q, k, v, o, do, lse, causal=causal, scale=scale)
    for _ in range(2):  # the built-in buffer keeps the previous call's contents
        got = noalloc_bwd(q, k, v, o, do, lse, causal, scale)
        assert api.device_status() == 0
        for g, w in zip(got, want):
            ref = w.double().cpu().numpy()
            assert rel_fro(g, ref) <= GRAD_RTOL


def test_noalloc_refuses_problems_beyond_the_buffer():
    # Delta and lse2 alone for Z*H*N = 2^24 rows need 128 MiB > 64 MiB.
    Z, H, N, D = 1024, 16, 1024, 64
    fake = 1 << 20  # never dereferenced: the size check runs before any launch
    rc = _native.lib().fa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                      Z, H, N, D, 0, 0.125, None)
    assert rc == _native.FA_ERR_SCRATCH_LIMIT
    assert "64 MiB" in _native.error_string(rc)
