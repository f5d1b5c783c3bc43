"""Pins of the oracle's masks (oracle/attn_oracle.c), each against something other
than the oracle's own formula.  zerotofrontier.app "FlashAttention", "Dropout,
block-sparsity, and other real-kernel details": sliding windows are functions of
(r, l) applied inside the tile, and a block mask marks whole tiles that are skipped.
Here key l is allowed for row r iff r + off - left <= l <= r + off + right (off =
Tk - Tq, -1 = unbounded side) and the 128-block (r // bs, l // bs) is marked."""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle


def draw(Tq, Tk, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((Tq, d)), rng.standard_normal((Tk, d)), rng.standard_normal((Tk, d)),
            rng.standard_normal((Tq, d)))


def band(Tq, Tk, left, right):
    """Allowed (r, l) of a window, from numpy's band routines: tril keeps l - r <= k,
    triu keeps l - r >= k, both offset by the bottom-right diagonal."""
    off = Tk - Tq
    m = np.ones((Tq, Tk), dtype=bool)
    if right >= 0:
        m &= np.tril(np.ones((Tq, Tk), dtype=bool), k=off + right)
    if left >= 0:
        m &= np.triu(np.ones((Tq, Tk), dtype=bool), k=off - left)
    return m


def sdpa(q, k, v, allowed, scale):
    """torch's scaled_dot_product_attention in float64 with a boolean mask, and lse from
    scipy's logsumexp; rows with no allowed key are returned as NaN (torch) and -inf."""
    t = [torch.tensor(x)[None, None] for x in (q, k, v)]
    o = torch.nn.functional.scaled_dot_product_attention(*t, attn_mask=torch.tensor(allowed)[None, None],
                                                         scale=scale)[0, 0].numpy()
    s = np.where(allowed, scale * q @ k.T, -np.inf)
    return o, logsumexp(s, axis=1)


def test_window_zero_is_the_diagonal_key():
    """window (0, 0): row r sees exactly key r + Tk - Tq, so O_r = V of that key and
    lse_r = c q_r . k_l; rows whose diagonal key does not exist see nothing."""
    for Tq, Tk in ((9, 9), (6, 11), (11, 6)):
        q, k, v, _ = draw(Tq, Tk, 5, Tq * Tk)
        o, lse = oracle.attention_fwd(q, k, v, False, 0.7, window=(0, 0))
        for r in range(Tq):
            l = r + Tk - Tq
            if 0 <= l < Tk:
                assert np.allclose(o[r], v[l], atol=1e-12) and abs(lse[r] - 0.7 * q[r] @ k[l]) < 1e-12
            else:
                assert np.all(o[r] == 0) and lse[r] == -np.inf


@pytest.mark.parametrize("Tq,Tk,left,right", [(40, 40, 7, 0), (40, 40, 5, 3), (30, 50, 12, -1), (50, 30, -1, 4),
                                              (33, 33, 0, 6), (20, 64, 9, 0)])
def test_window_matches_torch_sdpa(Tq, Tk, left, right):
    q, k, v, _ = draw(Tq, Tk, 8, Tq + 7 * Tk + left)
    allowed = band(Tq, Tk, left, right)
    o, lse = oracle.attention_fwd(q, k, v, False, 0.35, window=(left, right))
    o_ref, lse_ref = sdpa(q, k, v, allowed, 0.35)
    live = allowed.any(axis=1)
    assert np.allclose(o[live], o_ref[live], atol=1e-12)
    assert np.allclose(lse[live], lse_ref[live], atol=1e-12)
    assert np.all(o[~live] == 0) and np.all(lse[~live] == -np.inf)


def test_block_mask_all_ones_is_no_mask():
    q, k, v, _ = draw(300, 260, 16, 1)
    bm = np.ones((3, 3), dtype=np.uint8)
    for causal in (False, True):
        o1, l1 = oracle.attention_fwd(q, k, v, causal, 0.25)
        o2, l2 = oracle.attention_fwd(q, k, v, False, 0.25, window=(-1, 0) if causal else None, block_mask=bm)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_block_diagonal_mask_is_independent_blocks():
    """With only diagonal 128-blocks marked, each query block attends to its own key block:
    the same as separate unmasked problems on the blocks."""
    Tq = Tk = 300
    q, k, v, _ = draw(Tq, Tk, 8, 2)
    bm = np.eye(3, dtype=np.uint8)
    o, lse = oracle.attention_fwd(q, k, v, False, 0.5, block_mask=bm)
    for b in range(3):
        sl = slice(128 * b, min(Tq, 128 * (b + 1)))
        ob, lb = oracle.attention_fwd(q[sl], k[sl], v[sl], False, 0.5)
        assert np.allclose(o[sl], ob, atol=1e-13) and np.allclose(lse[sl], lb, atol=1e-13)


def test_block_mask_and_window_match_torch_sdpa():
    Tq, Tk, bs = 45, 70, 16
    q, k, v, _ = draw(Tq, Tk, 6, 3)
    rng = np.random.default_rng(4)
    bm = (rng.random((-(-Tq // bs), -(-Tk // bs))) < 0.6).astype(np.uint8)
    allowed = band(Tq, Tk, 20, 2) & np.kron(bm, np.ones((bs, bs)))[:Tq, :Tk].astype(bool)
    o, lse = oracle.attention_fwd(q, k, v, False, 0.4, window=(20, 2), block_mask=bm, block_size=bs)
    o_ref, lse_ref = sdpa(q, k, v, allowed, 0.4)
    live = allowed.any(axis=1)
    assert live.sum() > 10 and (~live).sum() > 0
    assert np.allclose(o[live], o_ref[live], atol=1e-12) and np.allclose(lse[live], lse_ref[live], atol=1e-12)
    assert np.all(o[~live] == 0) and np.all(lse[~live] == -np.inf)


def test_masked_gradients_match_torch_autograd():
    Tq, Tk, bs = 24, 40, 8
    q, k, v, do = draw(Tq, Tk, 4, 5)
    rng = np.random.default_rng(6)
    bm = (rng.random((3, 5)) < 0.7).astype(np.uint8)
    allowed = band(Tq, Tk, 10, 1) & np.kron(bm, np.ones((bs, bs)))[:Tq, :Tk].astype(bool)
    live = allowed.any(axis=1)
    g = oracle.attention_bwd(q, k, v, do, False, 0.6, window=(10, 1), block_mask=bm, block_size=bs)
    t = [torch.tensor(x, requires_grad=True) for x in (q, k, v)]
    o = torch.nn.functional.scaled_dot_product_attention(*(x[None, None] for x in t),
                                                         attn_mask=torch.tensor(allowed)[None, None], scale=0.6)[0, 0]
    (o[torch.tensor(live)] * torch.tensor(do)[torch.tensor(live)]).sum().backward()
    assert np.allclose(g["dq"][live], t[0].grad.numpy()[live], atol=1e-11)
    assert np.all(g["dq"][~live] == 0)
    assert np.allclose(g["dk"], t[1].grad.numpy(), atol=1e-11)
    assert np.allclose(g["dv"], t[2].grad.numpy(), atol=1e-11)


def test_masked_gradient_finite_differences():
    """Central differences of sum(O * dO) under a window and a block mask."""
    Tq, Tk, bs, h = 6, 7, 2, 1e-6
    q, k, v, do = draw(Tq, Tk, 3, 7)
    bm = np.array([[1, 1, 0, 1], [0, 1, 1, 1], [1, 0, 1, 1]], dtype=np.uint8)
    kw = dict(window=(3, 1), block_mask=bm, block_size=bs)
    g = oracle.attention_bwd(q, k, v, do, False, 0.9, **kw)

    def f(q, k, v):
        o, _ = oracle.attention_fwd(q, k, v, False, 0.9, **kw)
        return float((o * do).sum())

    for name, x, gx in (("q", q, g["dq"]), ("k", k, g["dk"]), ("v", v, g["dv"])):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            num[idx] = (f(**{**args, name: xp}) - f(**{**args, name: xm})) / (2 * h)
        assert np.allclose(num, gx, atol=2e-7), name
