"""Failure detection on the GPU, without faulting it.

A kernel wait that can never complete must give up after its bounded limit,
report FA_ERR_TIMEOUT (with the site of the wait) through the device status
word, and return normally: the context stays usable and the next calls run.
"""

import ctypes
import math

import pytest
import torch

from attention_sm_flashattention_gb300 import _native, api
from attention_sm_flashattention_gb300.inputs import make_inputs
from oracle import attention as orc

from helpers import O_ATOL, max_abs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    lib = _native.lib()
    torch.cuda.synchronize()
    assert api.device_status() == 0
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.fa_selftest_wait_timeout(stream) == _native.FA_OK
    raw = ctypes.c_int(0)
    rc = lib.fa_device_status_raw(stream, ctypes.byref(raw))
    assert rc == _native.FA_ERR_TIMEOUT
    assert raw.value & 0xFF == 1 and raw.value >> 8 == 200
    # the status word was cleared and the context still works
    assert api.device_status() == 0
    q, k, v, _ = make_inputs(1, 2, 256, 128, seed=77)
    o, lse = api.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    assert api.device_status() == 0
    o_ref, _ = orc.attn_fwd_ref(q, k, v, True, 1 / math.sqrt(128))
    assert max_abs(o, o_ref) <= O_ATOL
