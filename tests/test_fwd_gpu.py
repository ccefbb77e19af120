"""Forward parity: CUDA path (through the C ABI) against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

from attention_sm_flashattention_gb300 import api
from attention_sm_flashattention_gb300.inputs import make_inputs
from oracle import attention as orc

from helpers import LSE_ATOL, O_ATOL, max_abs

pytestmark = pytest.mark.gpu


def run_fwd(q, k, v, causal, scale):
    o, lse = api.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    assert api.device_status() == 0
    return o, lse


# Small shapes the oracle finishes in seconds: several query/key tiles and,
# for D = 256, the 64-key tiles whose causal diagonal spans two tiles.
SMALL = [
    (1, 2, 128, 64), (1, 1, 256, 64), (2, 3, 384, 64),
    (1, 1, 128, 128), (1, 2, 256, 128), (2, 2, 512, 128),
    (1, 1, 128, 256), (1, 2, 384, 256),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "z%dh%dn%dd%d" % s)
def test_fwd_small_full_compare(shape, causal):
    Z, H, N, D = shape
    q, k, v, _ = make_inputs(Z, H, N, D, seed=Z * 1000 + H * 100 + N + D + int(causal))
    scale = 1 / math.sqrt(D)
    o, lse = run_fwd(q, k, v, causal, scale)
    o_ref, lse_ref = orc.attn_fwd_ref(q, k, v, causal, scale)
    assert max_abs(o, o_ref) <= O_ATOL
    assert max_abs(lse, lse_ref) <= LSE_ATOL


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_zero_query_closed_form(D, causal):
    # Q = 0: every visible score is 0, O_i is the mean of the visible V rows.
    N = 256
    _, k, v, _ = make_inputs(1, 2, N, D, seed=5)
    q = torch.zeros_like(k)
    o, lse = run_fwd(q, k, v, causal, 1 / math.sqrt(D))
    vv = v.double().numpy()
    if causal:
        cnt = np.arange(1, N + 1)
        want = np.cumsum(vv, axis=2) / cnt[None, None, :, None]
        want_lse = np.broadcast_to(np.log(cnt), (1, 2, N))
    else:
        want = np.broadcast_to(vv.mean(axis=2, keepdims=True), vv.shape)
        want_lse = np.full((1, 2, N), math.log(N))
    assert max_abs(o, want) <= O_ATOL
    assert max_abs(lse, want_lse) <= LSE_ATOL


def test_fwd_causal_row0_is_v0():
    q, k, v, _ = make_inputs(1, 1, 256, 128, seed=9)
    o, lse = run_fwd(q, k, v, True, 0.0884)
    sc = float(np.float32(0.0884))
    assert max_abs(o[0, 0, 0], v[0, 0, 0].double().numpy()) <= 1e-3
    want = sc * float(q[0, 0, 0].double() @ k[0, 0, 0].double())
    assert abs(float(lse[0, 0, 0]) - want) <= LSE_ATOL


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_deterministic(causal):
    q, k, v, _ = make_inputs(2, 4, 512, 128, seed=11)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = api.fwd(q, k, v, causal=causal)
    o2, l2 = api.fwd(q, k, v, causal=causal)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fwd_writes_only_its_outputs():
    # Canary padding around the outputs must stay untouched.
    Z, H, N, D = 1, 3, 256, 128
    q, k, v, _ = make_inputs(Z, H, N, D, seed=12)
    pad = 4096
    o_buf = torch.full((pad * 2 + Z * H * N * D,), 7.0, dtype=torch.float16, device="cuda")
    l_buf = torch.full((pad * 2 + Z * H * N,), -3.0, dtype=torch.float32, device="cuda")
    o = o_buf[pad:pad + Z * H * N * D].view(Z, H, N, D)
    lse = l_buf[pad:pad + Z * H * N].view(Z, H, N)
    api.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, out=(o, lse))
    assert api.device_status() == 0
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    assert torch.all(l_buf[:pad] == -3.0) and torch.all(l_buf[-pad:] == -3.0)


def test_fwd_on_side_stream():
    q, k, v, _ = make_inputs(1, 2, 256, 64, seed=13)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = api.fwd(q.cuda(), k.cuda(), v.cuda(), causal=False)
    s.synchronize()
    o_ref, lse_ref = orc.attn_fwd_ref(q, k, v, False, 1 / 8)
    assert max_abs(o, o_ref) <= O_ATOL
