"""Every head of every benchmark workload against the fp64 oracle, through the
boundary's own calls: fa_fwd then fa_bwd (fp16), and fa_fwd_bf16 then
fa_bwd_bf16 for the bf16 runs, driven through ctypes with real device
buffers and a caller-allocated workspace.

The full-size workloads are the only runs that reach every wave of the
persistent schedules, so no head is left out: an error that corrupts one tile
of one late head fails here.  The oracle runs head by head on the host cores
(``oracle_pool``).  The Python API (``api.fwd`` / ``api.bwd``, what the
benchmark calls) must then give the same bits, since it launches the same
kernels through ``fa_fwd_ex`` / ``fa_bwd_ex``.
"""

import numpy as np
import pytest
import torch

from attention_sm_flashattention_gb300 import _native, api
from attention_sm_flashattention_gb300.inputs import WORKLOADS, make_inputs

from helpers import GRAD_RTOL, GRAD_RTOL_BF16, LSE_ATOL, O_ATOL, O_ATOL_BF16
from oracle_pool import FIELDS, all_head_errors

pytestmark = pytest.mark.gpu


def run_boundary(q, k, v, do, causal, scale, bf16):
    """fa_fwd and fa_bwd (or the bf16 pair) on device copies of the inputs,
    on torch's current stream.  Returns the device outputs."""
    lib = _native.lib()
    Z, H, N, D = q.shape
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((Z, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    need = lib.fa_bwd_workspace_size(Z, H, N, D, int(causal))
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    fwd, bwd = (lib.fa_fwd_bf16, lib.fa_bwd_bf16) if bf16 else (lib.fa_fwd, lib.fa_bwd)
    rc = fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(), Z, H, N, D, int(causal),
             scale, stream)
    assert rc == _native.FA_OK, _native.error_string(rc)
    rc = bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), dod.data_ptr(), lse.data_ptr(),
             dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), need, Z, H, N, D, int(causal), scale, stream)
    assert rc == _native.FA_OK, _native.error_string(rc)
    assert lib.fa_device_status(stream) == _native.FA_OK
    return (qd, kd, vd, dod), (o, lse, dq, dk, dv)


def host(t: torch.Tensor, heads: int) -> np.ndarray:
    """Flat-head host copy: fp16 stays fp16; bf16 becomes fp32 (exact)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.reshape(heads, *t.shape[2:]).numpy()


CASES = [(name, False) for name in WORKLOADS] + [("z128h8n1024d128", True), ("z128h8n1024d128c", True)]


@pytest.mark.parametrize("name,bf16", CASES, ids=[n + ("-bf16" if b else "") for n, b in CASES])
def test_workload_every_head(name, bf16):
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w.Z, w.H, w.N, w.D, seed=w.seed, dtype=torch.bfloat16 if bf16 else torch.float16)
    dev_in, dev_out = run_boundary(q, k, v, do, w.causal, w.scale, bf16)
    o, lse, dq, dk, dv = dev_out
    for t in dev_out:
        assert torch.isfinite(t).all()

    # the Python API launches the same kernels: identical bits
    qd, kd, vd, dod = dev_in
    o2, lse2 = api.fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq2, dk2, dv2 = api.bwd(qd, kd, vd, o2, dod, lse2, causal=w.causal, scale=w.scale)
    assert api.device_status() == 0
    for a, b in zip(dev_out, (o2, lse2, dq2, dk2, dv2)):
        assert torch.equal(a, b)

    nh = w.heads
    errs = all_head_errors(host(q, nh), host(k, nh), host(v, nh), host(do, nh), host(o, nh),
                           lse.detach().cpu().reshape(nh, w.N).numpy(), host(dq, nh), host(dk, nh), host(dv, nh),
                           w.causal, w.scale)
    assert not np.isnan(errs).any(), "some heads were not checked"
    o_tol = O_ATOL_BF16 if bf16 else O_ATOL
    g_tol = GRAD_RTOL_BF16 if bf16 else GRAD_RTOL
    limits = (o_tol, LSE_ATOL, g_tol, g_tol, g_tol)
    for f, (field, lim) in enumerate(zip(FIELDS, limits)):
        worst = int(np.argmax(errs[:, f]))
        assert errs[worst, f] <= lim, f"{name}: {field} {errs[worst, f]:.3e} > {lim:g} at head {worst}"
