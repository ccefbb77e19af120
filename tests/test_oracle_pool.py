"""The every-head comparison helper (``oracle_pool``) on the CPU: spawned
workers return each head's errors in the right row, and a mistake planted in
one head is reported at that head and no other."""

import numpy as np

from attention_sm_flashattention_gb300.inputs import make_inputs
from oracle import attention as orc
from oracle_pool import FIELDS, all_head_errors


def _oracle_outputs(q, k, v, do, causal, scale):
    o, lse = orc.attn_fwd_ref(q, k, v, causal, scale)
    dq, dk, dv = orc.attn_bwd_ref(q, k, v, do, causal, scale)
    return o, lse, dq, dk, dv


def test_pool_reports_each_head_in_its_row():
    Z, H, N, D, causal, scale = 2, 4, 128, 64, True, 0.125
    q, k, v, do = make_inputs(Z, H, N, D, seed=77)
    o, lse, dq, dk, dv = _oracle_outputs(q, k, v, do, causal, scale)
    heads = Z * H
    flat = lambda t: np.ascontiguousarray(np.asarray(t).reshape(heads, *np.asarray(t).shape[2:]))  # noqa: E731
    qn, kn, vn, don = (flat(t.numpy()) for t in (q, k, v, do))
    # outputs rounded as the GPU stores them, one head with a planted mistake
    o16, dq16, dk16, dv16 = (flat(t).astype(np.float16) for t in (o, dq, dk, dv))
    lse32 = flat(lse).astype(np.float32)
    bad = 5
    dk16[bad] = -dk16[bad]
    o16[bad, 3, 7] += np.float16(0.25)
    errs = all_head_errors(qn, kn, vn, don, o16, lse32, dq16, dk16, dv16, causal, scale, chunk=2)
    assert errs.shape == (heads, len(FIELDS))
    assert not np.isnan(errs).any()
    good = [h for h in range(heads) if h != bad]
    assert np.all(errs[good, 0] <= 2e-3) and np.all(errs[good, 1] <= 1e-4)
    assert np.all(errs[good, 2:] <= 1e-2)
    assert errs[bad, 0] > 0.2 and errs[bad, FIELDS.index("dk_rel_fro")] > 1.5
    assert errs[bad, FIELDS.index("dq_rel_fro")] <= 1e-2
