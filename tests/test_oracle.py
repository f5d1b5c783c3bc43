"""Pins for the fp64 oracle against what the pages and the mathematics fix.

Each check is chosen so that a plausible mistake in the oracle (a dropped
term, a wrong sign or index, a transposed operand, a wrong mask alignment, a
missing scale factor) fails at least one of them:

* the worked online-softmax example printed on the llmdeepdive 7.7 page;
* closed forms (one key, equal scores, causal row 0, a hand-worked causal
  d=1 case, bottom-right alignment for Tq != Tk, fully masked rows);
* invariants (P rows sum to 1, joint key/value permutation, shift and scale
  invariance, lse = logsumexp via scipy, exponents s - lse <= 0);
* the library routine the method reduces to (torch SDPA in float64 on CPU);
* central finite differences of the backward pass, and the gradient
  identities D_r = dO_r . O_r, sum_l dK_l = 0, sum_l dV_l = sum_r dO_r.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _mask(Tq, Tk, causal):
    r = np.arange(Tq)[:, None]
    l = np.arange(Tk)[None, :]
    return np.ones((Tq, Tk), bool) if not causal else (l <= r + (Tk - Tq))


# ---------------------------------------------------------------- worked example
def test_worked_example_online_softmax():
    g = json.load(open(os.path.join(GOLD, "online_softmax_worked_example.json")))
    pr, tol = g["printed"], g["printed_precision"]
    scores = [s for blk in g["blocks"] for s in blk]                 # [1, 3, 5]
    q = np.array([[1.0, 0.0, 0.0]])
    K = np.array([[s, 0.0, 0.0] for s in scores])
    V = np.eye(3)
    o, lse = oracle.attention_fwd(q, K, V, causal=False, scale=1.0)
    assert abs(o[0, 1] - pr["true_weight_of_3"]) <= tol
    ell = math.exp(lse[0] - max(scores))                             # l relative to the row max
    assert abs(ell - pr["ell_final"]) <= tol
    terms = [math.exp(s - max(scores)) for s in scores]
    for t, p in zip(terms, pr["direct_terms"]):
        assert abs(t - p) <= tol
    assert abs(lse[0] - math.log(sum(math.exp(s) for s in scores))) < 1e-14
    # the wrong turn: softmax of the first block alone
    o1, _ = oracle.attention_fwd(q, K[:2], V[:2, :], causal=False, scale=1.0)
    assert abs(o1[0, 1] - pr["local_softmax_weight_of_3"]) <= tol
    assert abs(o1[0, 1] - o[0, 1]) > 0.7


def test_worked_example_merge_trace():
    from oracle.tiled import flash_forward
    g = json.load(open(os.path.join(GOLD, "online_softmax_worked_example.json")))
    pr, tol = g["printed"], g["printed_precision"]
    q = np.array([[1.0, 0.0, 0.0]])
    K = np.array([[1.0, 0, 0], [3.0, 0, 0], [5.0, 0, 0]])
    res = flash_forward(q, K, np.eye(3), Br=1, Bc=2, scale=1.0, trace_row=0)
    b1, b2 = res.trace
    assert b1["m_new"] == pr["m_after_block_1"]
    assert abs(b1["ell"] - pr["ell_after_block_1"]) <= tol
    assert b2["m_old"] == pr["m_after_block_1"] and b2["m_new"] == pr["m_after_block_2"]
    assert abs(b2["ell_rescaled"] - pr["ell_rescaled_by_exp_minus_2"]) <= tol
    assert abs(b2["ell"] - pr["ell_final"]) <= tol
    assert abs(res.o[0, 1] - pr["true_weight_of_3"]) <= tol


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_single_key(causal):
    r = _rng(1)
    q, k, v = r.normal(size=(1, 5)), r.normal(size=(1, 5)), r.normal(size=(1, 5))
    o, lse = oracle.attention_fwd(q, k, v, causal, 0.3)
    np.testing.assert_array_equal(o, v)
    assert abs(lse[0] - 0.3 * float(q[0] @ k[0])) < 1e-15


def test_equal_scores_mean():
    r = _rng(2)
    Tq, Tk, d = 4, 9, 6
    v = r.normal(size=(Tk, d))
    o, lse = oracle.attention_fwd(np.zeros((Tq, d)), r.normal(size=(Tk, d)), v, False, 0.7)
    np.testing.assert_allclose(o, np.tile(v.mean(0), (Tq, 1)), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, math.log(Tk), rtol=0, atol=1e-15)
    # all keys equal: same weights, lse shifted by the common score
    q = r.normal(size=(Tq, d))
    k = np.tile(r.normal(size=(1, d)), (Tk, 1))
    o, lse = oracle.attention_fwd(q, k, v, False, 0.7)
    np.testing.assert_allclose(o, np.tile(v.mean(0), (Tq, 1)), atol=1e-14)
    np.testing.assert_allclose(lse, 0.7 * (q @ k[0]) + math.log(Tk), atol=1e-13)


def test_causal_row0_and_hand_case():
    r = _rng(3)
    q, k, v = r.normal(size=(6, 4)), r.normal(size=(6, 4)), r.normal(size=(6, 4))
    o, lse = oracle.attention_fwd(q, k, v, True, 0.5)
    np.testing.assert_array_equal(o[0], v[0])
    assert abs(lse[0] - 0.5 * float(q[0] @ k[0])) < 1e-15
    # d = 1, scores s_rl = k_l = ln(l + 1): weights 1 : 2 : 3 under the causal mask
    Q = np.ones((3, 1))
    K = np.log(np.array([[1.0], [2.0], [3.0]]))
    V = np.array([[1.0], [10.0], [100.0]])
    o, lse = oracle.attention_fwd(Q, K, V, True, 1.0)
    np.testing.assert_allclose(o[:, 0], [1.0, 7.0, 53.5], rtol=1e-15)
    np.testing.assert_allclose(lse, [0.0, math.log(3.0), math.log(6.0)], atol=1e-15)


def test_bottom_right_alignment_and_masked_rows():
    r = _rng(4)
    d = 3
    v = r.normal(size=(4, d))
    # Tq < Tk: row r sees keys l <= r + 2
    o, _ = oracle.attention_fwd(np.zeros((2, d)), r.normal(size=(4, d)), v, True, 1.0)
    np.testing.assert_allclose(o[0], v[:3].mean(0), atol=1e-15)
    np.testing.assert_allclose(o[1], v.mean(0), atol=1e-15)
    # Tq > Tk: rows 0 and 1 see no key at all
    v2 = r.normal(size=(2, d))
    o, lse = oracle.attention_fwd(np.zeros((4, d)), r.normal(size=(2, d)), v2, True, 1.0)
    np.testing.assert_array_equal(o[:2], 0.0)
    assert np.all(lse[:2] == -np.inf)
    np.testing.assert_allclose(o[2], v2[0], atol=0)
    np.testing.assert_allclose(o[3], v2.mean(0), atol=1e-15)
    out = oracle.attention_bwd(np.zeros((4, d)), r.normal(size=(2, d)), v2, r.normal(size=(4, d)),
                               True, 1.0)
    np.testing.assert_array_equal(out["dq"][:2], 0.0)


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal,Tq,Tk", [(False, 5, 7), (True, 7, 7), (True, 5, 7), (True, 7, 5)])
def test_probability_rows(causal, Tq, Tk):
    r = _rng(5)
    q, k = r.normal(size=(Tq, Tk)), r.normal(size=(Tk, Tk))
    P, lse = oracle.attention_fwd(q, k, np.eye(Tk), causal, 0.9)    # V = I makes O = P
    live = np.isfinite(lse)
    np.testing.assert_allclose(P[live].sum(1), 1.0, atol=1e-14)
    assert np.all(P >= 0)
    assert np.all(P[~_mask(Tq, Tk, causal)] == 0.0)
    s = 0.9 * q @ k.T
    s[~_mask(Tq, Tk, causal)] = -np.inf
    np.testing.assert_allclose(lse[live], logsumexp(s[live], axis=1), atol=1e-13)
    assert np.all(s[live] - lse[live][:, None] <= 1e-13)


def test_permutation_shift_scale():
    r = _rng(6)
    Tq, Tk, d = 8, 11, 5
    q, k, v = r.normal(size=(Tq, d)), r.normal(size=(Tk, d)), r.normal(size=(Tk, d))
    o, lse = oracle.attention_fwd(q, k, v, False, 0.4)
    perm = r.permutation(Tk)
    o2, lse2 = oracle.attention_fwd(q, k[perm], v[perm], False, 0.4)
    np.testing.assert_allclose(o2, o, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, atol=1e-14)
    u = r.normal(size=(d,))
    o3, lse3 = oracle.attention_fwd(q, k + u, v, False, 0.4)       # every score of row r moves by c q_r.u
    np.testing.assert_allclose(o3, o, atol=1e-13)
    np.testing.assert_allclose(lse3, lse + 0.4 * (q @ u), atol=1e-13)
    o4, _ = oracle.attention_fwd(q, k, -2.5 * v, False, 0.4)
    np.testing.assert_allclose(o4, -2.5 * o, atol=1e-14)
    assert np.all(o <= v.max(0) + 1e-15) and np.all(o >= v.min(0) - 1e-15)


@pytest.mark.parametrize("causal,Tq,Tk", [(False, 13, 17), (True, 16, 16), (True, 9, 21), (True, 21, 9)])
def test_matches_torch_sdpa_float64(causal, Tq, Tk):
    r = _rng(7)
    d = 6
    q, k, v = r.normal(size=(Tq, d)), r.normal(size=(Tk, d)), r.normal(size=(Tk, d))
    o, lse = oracle.attention_fwd(q, k, v, causal, 0.35)
    m = torch.from_numpy(_mask(Tq, Tk, causal))
    live = m.any(1).numpy()
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=m[None], scale=0.35)[0].numpy()
    np.testing.assert_allclose(o[live], ref[live], atol=1e-13)
    # rows subset equals the corresponding full rows
    rows = np.array([Tq - 1, 0, Tq // 2])
    o_s, lse_s = oracle.attention_fwd(q, k, v, causal, 0.35, rows=rows)
    np.testing.assert_array_equal(o_s, o[rows])
    np.testing.assert_array_equal(lse_s, lse[rows])


# ---------------------------------------------------------------- backward
def _loss(q, k, v, dO, causal, scale):
    o, _ = oracle.attention_fwd(q, k, v, causal, scale, nthreads=1)
    return float((o * dO).sum())


@pytest.mark.parametrize("causal,Tq,Tk", [(False, 5, 6), (True, 6, 6), (True, 4, 7), (True, 7, 4)])
def test_backward_finite_differences(causal, Tq, Tk):
    r = _rng(8)
    d, c, h = 3, 0.8, 1e-6
    q, k, v, dO = (r.normal(size=s) for s in [(Tq, d), (Tk, d), (Tk, d), (Tq, d)])
    g = oracle.attention_bwd(q, k, v, dO, causal, c, nthreads=2)
    for name, x, grad in (("q", q, g["dq"]), ("k", k, g["dk"]), ("v", v, g["dv"])):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], dO, causal, c)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], dO, causal, c)
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - grad).max() / max(1.0, np.abs(grad).max())
        assert err < 1e-7, (name, err)


@pytest.mark.parametrize("causal,Tq,Tk", [(False, 19, 23), (True, 24, 24), (True, 10, 30), (True, 30, 10)])
def test_backward_identities_and_torch(causal, Tq, Tk):
    r = _rng(9)
    d, c = 5, 0.45
    q, k, v, dO = (r.normal(size=s) for s in [(Tq, d), (Tk, d), (Tk, d), (Tq, d)])
    g = oracle.attention_bwd(q, k, v, dO, causal, c, want_o=True)
    o, lse = oracle.attention_fwd(q, k, v, causal, c)
    np.testing.assert_allclose(g["o"], o, atol=1e-14)
    np.testing.assert_allclose(g["lse"], lse, atol=1e-14)
    live = np.isfinite(lse)
    np.testing.assert_allclose(g["D"], (dO * o).sum(1), atol=1e-13)       # D_r = dO_r . O_r
    np.testing.assert_allclose(g["dk"].sum(0), 0.0, atol=1e-12)           # sum_l dS_rl = 0
    np.testing.assert_allclose(g["dv"].sum(0), dO[live].sum(0), atol=1e-12)
    # torch autograd on the float64 library attention
    m = torch.from_numpy(_mask(Tq, Tk, causal))
    tq, tk, tv = (torch.from_numpy(x).clone().requires_grad_(True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None],
                                                           attn_mask=m[None], scale=c)[0]
    out = torch.where(torch.from_numpy(live)[:, None], out, torch.zeros_like(out))
    (out * torch.from_numpy(dO)).sum().backward()
    np.testing.assert_allclose(g["dq"], tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(g["dk"], tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(g["dv"], tv.grad.numpy(), atol=1e-12)
    # row/key subsets equal the corresponding full entries
    rows, keys = np.array([Tq - 1, 2]), np.array([0, Tk - 1, Tk // 3])
    gs = oracle.attention_bwd(q, k, v, dO, causal, c, rows=rows, keys=keys, nthreads=3)
    np.testing.assert_allclose(gs["dq"], g["dq"][rows], atol=1e-15)
    np.testing.assert_allclose(gs["dk"], g["dk"][keys], atol=1e-15)
    np.testing.assert_allclose(gs["dv"], g["dv"][keys], atol=1e-15)


def test_thread_count_does_not_change_results():
    r = _rng(10)
    q, k, v, dO = (r.normal(size=(33, 7)) for _ in range(4))
    a = oracle.attention_bwd(q, k, v, dO, True, 0.3, nthreads=1)
    b = oracle.attention_bwd(q, k, v, dO, True, 0.3, nthreads=5)
    for n in ("dq", "dk", "dv", "lse", "D"):
        np.testing.assert_array_equal(a[n], b[n])
