"""Pins for the fp64 oracle, all on the CPU.

The oracle is checked against things other than itself: closed forms,
invariants the mathematics fixes, pure-Python brute force, central finite
differences of the loss ``L = sum(O * dO)`` and an independent library
(torch's fp64 CPU ``scaled_dot_product_attention`` with autograd).  The last
block plants plausible mistakes in copies of the oracle and checks that at
least one pin catches each of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from attention_sm_flashattention_gb300.inputs import WORKLOADS, make_inputs
from oracle import attention as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_head(n, d, seed, n_k=None):
    rng = np.random.default_rng(seed)
    n_k = n if n_k is None else n_k
    q = rng.standard_normal((n, d))
    k = rng.standard_normal((n_k, d))
    v = rng.standard_normal((n_k, d))
    do = rng.standard_normal((n, d))
    return q, k, v, do


# ---------------------------------------------------------------- closed forms


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 4), (7, 3), (64, 16), (128, 64)])
def test_zero_query_closed_form(causal, n, d):
    # Q = 0 makes every unmasked score 0: O_i is the mean of the visible V rows
    # and lse_i = log(#visible keys).
    _, k, v, _ = rand_head(n, d, 1)
    q = np.zeros((n, d))
    o, lse = orc.attn_fwd_head(q, k, v, causal, 0.125)
    if causal:
        counts = np.arange(1, n + 1)
        want_o = np.cumsum(v, axis=0) / counts[:, None]
        want_lse = np.log(counts)
    else:
        want_o = np.broadcast_to(v.mean(axis=0), (n, d))
        want_lse = np.full(n, math.log(n))
    np.testing.assert_allclose(o, want_o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-13)


@pytest.mark.parametrize("n,d", [(2, 8), (33, 16)])
def test_causal_row0(n, d):
    # Row 0 of a causal head sees key 0 only: O_0 = V_0, lse_0 = scale q0.k0.
    q, k, v, _ = rand_head(n, d, 2)
    sc = float(np.float32(0.3))
    o, lse = orc.attn_fwd_head(q, k, v, True, sc)
    np.testing.assert_allclose(o[0], v[0], rtol=0, atol=1e-14)
    assert lse[0] == pytest.approx(sc * float(q[0] @ k[0]), abs=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v(causal):
    n, d = 40, 12
    q, k, _, _ = rand_head(n, d, 3)
    c = np.linspace(-2, 3, d)
    v = np.broadcast_to(c, (n, d)).copy()
    o, _ = orc.attn_fwd_head(q, k, v, causal, 0.5)
    np.testing.assert_allclose(o, np.broadcast_to(c, (n, d)), rtol=0, atol=1e-13)


def test_single_key():
    q, k, v, _ = rand_head(1, 9, 4)
    sc = float(np.float32(0.7))
    o, lse = orc.attn_fwd_head(q, k, v, False, sc)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
    assert lse[0] == pytest.approx(sc * float(q[0] @ k[0]), abs=1e-14)


# ------------------------------------------------------------------ invariants


@pytest.mark.parametrize("causal", [False, True])
def test_prob_rows_sum_to_one_and_mask(causal):
    q, k, _, _ = rand_head(50, 16, 5)
    p, lse = orc.softmax_probs(orc.scores(q, k, 0.25, causal))
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(p >= 0)
    if causal:
        assert np.all(np.triu(p, 1) == 0.0)
        assert np.all(np.diag(p) > 0)
    # P_ij = exp(S_ij - lse_i): the row statistic regenerates P (the backward's
    # recompute relies on this).
    s = orc.scores(q, k, 0.25, causal)
    np.testing.assert_allclose(np.exp(s - lse[:, None]), p, rtol=1e-13, atol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sum_invariants(causal):
    q, k, v, do = rand_head(48, 16, 6)
    dq, dk, dv = orc.attn_bwd_head(q, k, v, do, causal, 0.25)
    # rows of P sum to 1  =>  sum_j dV_j = sum_j (P^T dO)_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), rtol=0, atol=1e-12)
    # rows of dS sum to 0  =>  sum_j dK_j = scale * sum_i (sum_j dS_ij) Q_i = 0
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, rtol=0, atol=1e-12)


def test_delta_identity():
    # Delta = rowsum(O * dO) (the form §二 writes) equals rowsum(P * dP).
    q, k, v, do = rand_head(30, 8, 7)
    p, _ = orc.softmax_probs(orc.scores(q, k, 0.4, False))
    o = p @ v
    lhs = np.sum(o * do, axis=1)
    rhs = np.sum(p * (do @ v.T), axis=1)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-13, atol=1e-13)


def test_kv_permutation_invariance():
    q, k, v, do = rand_head(24, 8, 8)
    perm = np.random.default_rng(0).permutation(24)
    o1, l1 = orc.attn_fwd_head(q, k, v, False, 0.3)
    o2, l2 = orc.attn_fwd_head(q, k[perm], v[perm], False, 0.3)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
    _, dk1, dv1 = orc.attn_bwd_head(q, k, v, do, False, 0.3)
    _, dk2, dv2 = orc.attn_bwd_head(q, k[perm], v[perm], do, False, 0.3)
    np.testing.assert_allclose(dk1[perm], dk2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv1[perm], dv2, rtol=0, atol=1e-12)


def test_shift_invariance_of_o():
    # Adding the same vector c to every key adds scale*(q_i.c) to every score
    # of row i: P (hence O) is unchanged and lse_i moves by exactly that.
    q, k, v, _ = rand_head(20, 6, 9)
    c = np.random.default_rng(1).standard_normal(6)
    o1, l1 = orc.attn_fwd_head(q, k, v, False, 0.5)
    o2, l2 = orc.attn_fwd_head(q, k + c, v, False, 0.5)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, 0.5 * (q @ c), rtol=0, atol=1e-12)


# ----------------------------------------------------------------- brute force


def brute_force_fwd(q, k, v, causal, scale):
    n, d = len(q), len(q[0])
    o, lse = [], []
    for i in range(n):
        s = []
        for j in range(len(k)):
            if causal and j > i:
                continue
            s.append((j, scale * sum(q[i][t] * k[j][t] for t in range(d))))
        mx = max(x for _, x in s)
        w = [(j, math.exp(x - mx)) for j, x in s]
        tot = sum(x for _, x in w)
        o.append([sum(x * v[j][t] for j, x in w) / tot for t in range(d)])
        lse.append(mx + math.log(tot))
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 1), (3, 2), (8, 5)])
def test_brute_force(causal, n, d):
    q, k, v, _ = rand_head(n, d, 10 + n)
    sc = float(np.float32(1 / math.sqrt(d)))
    want_o, want_lse = brute_force_fwd(q.tolist(), k.tolist(), v.tolist(), causal, sc)
    o, lse = orc.attn_fwd_head(q, k, v, causal, sc)
    np.testing.assert_allclose(o, np.array(want_o), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, np.array(want_lse), rtol=1e-13, atol=1e-14)


# ------------------------------------------------------- finite differences


def fd_grads(fwd, q, k, v, do, causal, scale, h=1e-6):
    """Central differences of L = sum(O * dO) with respect to q, k and v."""
    grads = []
    for which in range(3):
        base = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(base[which])
        for idx in np.ndindex(*g.shape):
            plus = [t.copy() for t in base]
            minus = [t.copy() for t in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            lp = np.sum(fwd(*plus, causal, scale)[0] * do)
            lm = np.sum(fwd(*minus, causal, scale)[0] * do)
            g[idx] = (lp - lm) / (2 * h)
        grads.append(g)
    return grads


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(5, 3), (16, 16)])
def test_finite_differences(causal, n, d):
    q, k, v, do = rand_head(n, d, 20 + n)
    sc = float(np.float32(1 / math.sqrt(d)))
    got = orc.attn_bwd_head(q, k, v, do, causal, sc)
    want = fd_grads(orc.attn_fwd_head, q, k, v, do, causal, sc)
    for g, w in zip(got, want):
        rel = np.linalg.norm(g - w) / np.linalg.norm(w)
        assert rel <= 1e-6, rel


# ------------------------------------------------------ independent library


def torch_sdpa(q, k, v, do, causal, scale):
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk[None], tv[None], is_causal=causal, scale=scale)[0]
    o.backward(torch.tensor(do, dtype=torch.float64))
    s = (tq @ tk.T).detach() * scale
    if causal:
        s = s.masked_fill(torch.ones_like(s, dtype=torch.bool).triu(1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return (o.detach().numpy(), lse.numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy())


@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_sdpa_small_workload(causal):
    w = WORKLOADS["z1h2n128d64"]
    q, k, v, do = make_inputs(w.Z, w.H, w.N, w.D, w.seed)
    o, lse = orc.attn_fwd_ref(q, k, v, causal, w.scale)
    dq, dk, dv = orc.attn_bwd_ref(q, k, v, do, causal, w.scale)
    sc = float(np.float32(w.scale))
    for h in range(w.H):
        args = [t[0, h].double().numpy() for t in (q, k, v, do)]
        t_o, t_lse, t_dq, t_dk, t_dv = torch_sdpa(*args, causal, sc)
        np.testing.assert_allclose(o[0, h], t_o, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], t_lse, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dq[0, h], t_dq, rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(dk[0, h], t_dk, rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(dv[0, h], t_dv, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_sdpa_n256_slice(causal):
    q, k, v, do = make_inputs(1, 1, 256, 128, 77)
    sc = 1 / math.sqrt(128)
    o, lse = orc.attn_fwd_ref(q, k, v, causal, sc)
    grads = orc.attn_bwd_ref(q, k, v, do, causal, sc)
    args = [t[0, 0].double().numpy() for t in (q, k, v, do)]
    want = torch_sdpa(*args, causal, float(np.float32(sc)))
    got = (o[0, 0], lse[0, 0]) + tuple(g[0, 0] for g in grads)
    for g, w_ in zip(got, want):
        np.testing.assert_allclose(g, w_, rtol=1e-10, atol=1e-11)


def test_heads_subset_matches_full():
    q, k, v, do = make_inputs(2, 3, 32, 16, 5)
    o, lse = orc.attn_fwd_ref(q, k, v, True, 0.25)
    o_s, lse_s = orc.attn_fwd_ref(q, k, v, True, 0.25, heads=[4, 1])
    np.testing.assert_array_equal(o_s[0], o.reshape(6, 32, 16)[4])
    np.testing.assert_array_equal(lse_s[1], lse.reshape(6, 32)[1])
    g = orc.attn_bwd_ref(q, k, v, do, True, 0.25)
    g_s = orc.attn_bwd_ref(q, k, v, do, True, 0.25, heads=[5])
    for a, b in zip(g, g_s):
        np.testing.assert_array_equal(b[0], a.reshape(6, 32, 16)[5])


# ---------------------------------------------------------- page-printed data


def test_causal_tile_count_golden():
    g = json.load(open(os.path.join(GOLDEN, "causal_tiles.json")))
    t = g["n_tiles"]
    assert orc.causal_tile_count(t, False) == g["non_causal_tiles"]
    assert orc.causal_tile_count(t, True) == g["causal_tiles"]
    saved = 100.0 * (1 - g["causal_tiles"] / g["non_causal_tiles"])
    assert saved == pytest.approx(g["saving_percent"], abs=1e-12)


# ---------------------------------------------------------- planted mistakes


def _mutant_bwd(kind):
    def bwd(q, k, v, do, causal, scale):
        s = orc.scores(q, k, scale, causal)
        p, _ = orc.softmax_probs(s)
        dp = do @ v.T
        delta = np.sum(p * dp, axis=1, keepdims=True)
        if kind == "no_scale":
            ds = p * (dp - delta)
        elif kind == "no_delta":
            ds = scale * p * dp
        else:
            ds = scale * p * (dp - delta)
        dq = ds @ k
        dk = ds @ q if kind == "dk_untransposed" else ds.T @ q
        dv = p @ do if kind == "dv_untransposed" else p.T @ do
        return dq, dk, dv
    return bwd


@pytest.mark.parametrize("kind", ["no_scale", "no_delta", "dk_untransposed", "dv_untransposed"])
def test_pins_catch_planted_backward_mistakes(kind):
    q, k, v, do = rand_head(6, 4, 30)
    got = _mutant_bwd(kind)(q, k, v, do, False, 0.5)
    want = fd_grads(orc.attn_fwd_head, q, k, v, do, False, 0.5)
    worst = max(np.linalg.norm(g - w) / np.linalg.norm(w) for g, w in zip(got, want))
    assert worst > 1e-3


def test_pins_catch_planted_forward_mistakes():
    n, d = 8, 4
    q, k, v, _ = rand_head(n, d, 31)
    sc = 0.5
    # (a) mask that also hides the diagonal's neighbour the wrong way (j >= i)
    s = (q @ k.T) * sc
    bad = np.where(np.arange(n)[None, :] < np.arange(n)[:, None], -np.inf, s)
    p, _ = orc.softmax_probs(bad)
    assert not np.allclose((p @ v)[0], v[0])
    # (b) lse without the max term fails the N = 1 closed form
    lse_bad = np.log(np.sum(np.exp(s[:1, :1] - s[:1, :1])))
    assert abs(lse_bad - sc * float(q[0] @ k[0])) > 1e-6
    # (c) scaling after the softmax instead of before changes O
    p_good, _ = orc.softmax_probs(s)
    p_late, _ = orc.softmax_probs(q @ k.T)
    assert not np.allclose(p_good @ v, p_late @ v)


def test_bf16_inputs_widen_exactly():
    # bf16 carries 8 significant bits: these values are exact in bf16 and
    # must reach the oracle unchanged.
    vals = [1.0, 1.0 + 2.0 ** -7, -3.0, 2.0 ** -20, 1.5 * 2.0 ** 60]
    t = torch.tensor(vals, dtype=torch.bfloat16)
    assert list(orc._f64(t)) == vals


def test_bf16_closed_form_zero_q():
    # Q = 0 in bf16: every row of P is uniform, O_i = mean_j V_j and
    # lse_i = ln N, whatever the (bf16) K and V.
    n, d = 64, 16
    g = torch.Generator().manual_seed(5)
    q = torch.zeros(1, 1, n, d, dtype=torch.bfloat16)
    k = torch.randn(1, 1, n, d, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 1, n, d, generator=g).to(torch.bfloat16)
    o, lse = orc.attn_fwd_ref(q, k, v, False, 0.25)
    vm = v.float().double().numpy()[0, 0].mean(axis=0)
    assert np.max(np.abs(o[0, 0] - vm)) < 1e-14
    assert np.max(np.abs(lse - np.log(n))) < 1e-14


# ------------------------------------ grouped K/V heads, unequal/ragged lengths


def rand_gqa(z, h, h_kv, n_q, n_k, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((z, h, n_q, d))
    k = rng.standard_normal((z, h_kv, n_k, d))
    v = rng.standard_normal((z, h_kv, n_k, d))
    do = rng.standard_normal((z, h, n_q, d))
    return q, k, v, do


def brute_force_fwd_offset(q, k, v, causal, scale):
    """Pure-Python loops: query i is position len(k) - len(q) + i of the sequence."""
    n_q, n_k, d = len(q), len(k), len(q[0])
    o, lse = [], []
    for i in range(n_q):
        pos = n_k - n_q + i
        s = [(j, scale * sum(q[i][t] * k[j][t] for t in range(d))) for j in range(n_k) if not (causal and j > pos)]
        mx = max(x for _, x in s)
        w = [(j, math.exp(x - mx)) for j, x in s]
        tot = sum(x for _, x in w)
        o.append([sum(x * v[j][t] for j, x in w) / tot for t in range(d)])
        lse.append(mx + math.log(tot))
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n_q,n_k,d", [(1, 1, 2), (1, 7, 3), (3, 8, 2), (5, 6, 4), (6, 3, 2)])
def test_brute_force_unequal_lengths(causal, n_q, n_k, d):
    q, k, v, _ = rand_head(n_q, d, 40 + n_q + n_k, n_k=n_k)
    sc = float(np.float32(1 / math.sqrt(d)))
    if causal and n_q > n_k:
        with pytest.raises(ValueError):
            orc.attn_fwd_head(q, k, v, causal, sc)
        return
    want_o, want_lse = brute_force_fwd_offset(q.tolist(), k.tolist(), v.tolist(), causal, sc)
    o, lse = orc.attn_fwd_head(q, k, v, causal, sc)
    np.testing.assert_allclose(o, np.array(want_o), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, np.array(want_lse), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("n_q,n_k", [(1, 9), (5, 12), (130, 300)])
def test_zero_query_closed_form_offset(n_q, n_k):
    # Q = 0, causal, queries at the end: query i sees keys 0..i + n_k - n_q,
    # so O_i is the mean of those V rows and lse_i the log of their count.
    d = 6
    _, k, v, _ = rand_head(n_q, d, 50, n_k=n_k)
    o, lse = orc.attn_fwd_head(np.zeros((n_q, d)), k, v, True, 0.3)
    counts = np.arange(n_q) + (n_k - n_q) + 1
    np.testing.assert_allclose(o, (np.cumsum(v, axis=0) / np.arange(1, n_k + 1)[:, None])[counts - 1],
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.log(counts), rtol=0, atol=1e-13)


def test_decode_row_sees_whole_context():
    # One query at the end of the sequence: causal and non-causal agree.
    q, k, v, do = rand_head(1, 16, 51, n_k=37)
    for a, b in zip(orc.attn_fwd_head(q, k, v, True, 0.25), orc.attn_fwd_head(q, k, v, False, 0.25)):
        np.testing.assert_array_equal(a, b)
    for a, b in zip(orc.attn_bwd_head(q, k, v, do, True, 0.25), orc.attn_bwd_head(q, k, v, do, False, 0.25)):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n_q,n_k", [(4, 6), (5, 5)])
def test_finite_differences_grouped(causal, n_q, n_k):
    # Two K/V heads each shared by two query heads: the gradient of a shared
    # K or V is the derivative of the total loss over all four query heads.
    q, k, v, do = rand_gqa(1, 4, 2, n_q, n_k, 3, 52 + n_q)
    sc = float(np.float32(0.6))
    got = orc.attn_bwd_ref(q, k, v, do, causal, sc)
    want = fd_grads(lambda a, b, c, cz, s: orc.attn_fwd_ref(a, b, c, cz, s), q, k, v, do, causal, sc)
    for g, w in zip(got, want):
        rel = np.linalg.norm(g - w) / np.linalg.norm(w)
        assert rel <= 1e-6, rel


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("h,h_kv,n_q,n_k", [(4, 2, 16, 24), (8, 1, 9, 9), (6, 3, 130, 257)])
def test_against_torch_sdpa_grouped(causal, h, h_kv, n_q, n_k):
    # torch's enable_gqa shares K/V head h // g among query heads h, and its
    # causal_lower_right bias aligns the causal diagonal to the last query
    # with the last key; both are the library's own definitions.
    from torch.nn.attention.bias import causal_lower_right
    q, k, v, do = rand_gqa(2, h, h_kv, n_q, n_k, 8, 53 + h)
    sc = float(np.float32(0.35))
    o, lse = orc.attn_fwd_ref(q, k, v, causal, sc)
    dq, dk, dv = orc.attn_bwd_ref(q, k, v, do, causal, sc)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    mask = causal_lower_right(n_q, n_k) if causal else None
    t_o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=sc, enable_gqa=True)
    t_o.backward(torch.tensor(do))
    np.testing.assert_allclose(o, t_o.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-11)
    # lse: the log-sum-exp of torch's own masked scores
    s = torch.einsum("zhqd,zhkd->zhqk", torch.tensor(q), torch.tensor(k).repeat_interleave(h // h_kv, dim=1)) * sc
    if causal:
        s = s.masked_fill(~causal_lower_right(n_q, n_k)._materialize(), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=1e-12, atol=1e-12)


def test_grouped_heads_subset_matches_full():
    q, k, v, do = rand_gqa(2, 6, 2, 12, 20, 4, 54)
    o, lse = orc.attn_fwd_ref(q, k, v, True, 0.4)
    o_s, _ = orc.attn_fwd_ref(q, k, v, True, 0.4, heads=[7, 2])
    np.testing.assert_array_equal(o_s[0], o.reshape(12, 12, 4)[7])
    dq, dk, dv = orc.attn_bwd_ref(q, k, v, do, True, 0.4)
    heads = [7, 2, 8]
    assert orc.sampled_kv_heads(heads, 3) == [2, 0]
    dq_s, dk_s, dv_s = orc.attn_bwd_ref(q, k, v, do, True, 0.4, heads=heads)
    np.testing.assert_array_equal(dq_s[2], dq.reshape(12, 12, 4)[8])
    np.testing.assert_array_equal(dk_s[0], dk.reshape(4, 20, 4)[2])
    np.testing.assert_array_equal(dv_s[1], dv.reshape(4, 20, 4)[0])


def test_pins_catch_planted_grouping_and_alignment_mistakes():
    from torch.nn.attention.bias import causal_lower_right
    q, k, v, do = rand_gqa(1, 4, 2, 3, 5, 4, 55)
    sc = 0.5
    # (a) query head h reading K/V head h % H_kv instead of h // g
    o_good, _ = orc.attn_fwd_ref(q, k, v, False, sc)
    o_bad = np.stack([orc.attn_fwd_head(q[0, hh], k[0, hh % 2], v[0, hh % 2], False, sc)[0] for hh in range(4)])
    t_o = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), torch.tensor(k), torch.tensor(v), scale=sc, enable_gqa=True).numpy()
    assert np.allclose(o_good[0], t_o[0]) and not np.allclose(o_bad, t_o[0])
    # (b) causal diagonal aligned to the first query instead of the last
    s = (q[0, 0] @ k[0, 0].T) * sc
    top_left = np.where(np.arange(5)[None, :] > np.arange(3)[:, None], -np.inf, s)
    p_bad, _ = orc.softmax_probs(top_left)
    t_o = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q[:, :1]), torch.tensor(k[:, :1]), torch.tensor(v[:, :1]), scale=sc,
        attn_mask=causal_lower_right(3, 5)).numpy()[0, 0]
    assert not np.allclose(p_bad @ v[0, 0], t_o)
    np.testing.assert_allclose(orc.attn_fwd_head(q[0, 0], k[0, 0], v[0, 0], True, sc)[0], t_o, rtol=1e-12)
    # (c) dK of a shared head taken from one query head only
    dk_one = orc.attn_bwd_head(q[0, 0], k[0, 0], v[0, 0], do[0, 0], False, sc)[1]
    assert not np.allclose(dk_one, orc.attn_bwd_ref(q, k, v, do, False, sc)[1][0, 0])
