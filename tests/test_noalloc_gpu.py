"""fa_bwd_noalloc: the backward with its scratch in the library's static
device buffer computes exactly what fa_bwd computes (same kernels, outputs
equal bit for bit), and refuses problems whose scratch does not fit before
enqueueing anything.
"""

import math

import pytest
import torch

from attention_sm_flashattention_gb300 import _native, api
from attention_sm_flashattention_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_equals_bwd(D, causal):
    Z, H, N = 2, 3, 300
    q, k, v, do = (t.cuda() for t in make_inputs(Z, H, N, D, seed=880 + D + int(causal)))
    scale = 1 / math.sqrt(D)
    o, lse = api.fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = api.bwd(q, k, v, o, do, lse, causal=causal, scale=scale)
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = _native.lib().fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                      lse.data_ptr(), dq2.data_ptr(), dk2.data_ptr(), dv2.data_ptr(), Z, H, N, D,
                                      int(causal), scale, torch.cuda.current_stream().cuda_stream)
    assert rc == _native.FA_OK
    assert api.device_status() == 0
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_noalloc_refuses_scratch_past_its_buffer():
    # 64 x 128 heads of 1152 rows need 2 x 36 MiB of scratch, more than the
    # 64 MiB buffer: refused on the host, so the (never dereferenced)
    # addresses below are never handed to a kernel.
    fake = 1 << 20
    Z, H, N, D = 64, 128, 1152, 128
    assert _native.lib().fa_bwd_workspace_size(Z, H, N, D, 0) > _native.FA_NOALLOC_SCRATCH_BYTES
    rc = _native.lib().fa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, Z, H, N, D, 0, 0.125,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == _native.FA_ERR_SCRATCH_LIMIT
    assert api.device_status() == 0
