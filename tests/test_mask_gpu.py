"""Sliding windows and block masks (fa_fwd_masked) against the fp64 oracle under the
same mask.  zerotofrontier.app "FlashAttention", "Dropout, block-sparsity, and other
real-kernel details": windows are functions of (r, l) computed inside the tile, and
tiles a block mask marks empty are skipped exactly as causal tiles are.  Every element
for ragged shapes at d = 64, 128, 256; the causal window through the masked entry point
is bitwise fa_fwd; a sliding window on the 4096/d128 workload, sampled heads."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_05_gb300 import inputs
from gpu_util import TOL_GRAD, TOL_LSE, TOL_O_BF16, fwd_errors, half_ulp_bf16, heads_of, rows_of, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_io_aware_05_gb300 import fa as _fa
    return _fa


def random_mask(B, H, Tq, Tk, per_head, seed, density=0.6):
    g = torch.Generator().manual_seed(seed)
    shape = (B, H, -(-Tq // 128), -(-Tk // 128)) if per_head else (-(-Tq // 128), -(-Tk // 128))
    m = (torch.rand(shape, generator=g) < density).to(torch.uint8)
    if m.dim() == 2:
        m[0] = 0                               # a query block with no key block at all
    else:
        m[0, 0, 0] = 0
    return m


def check(fa, w, window, bmask, heads, rows=None):
    x = inputs.generate(w, with_grad=False, device="cuda")
    bm_dev = None if bmask is None else bmask.to("cuda")
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], False, w.scale, window=window, block_mask=bm_dev)
    assert fa.fa_sync_status() == fa.FA_OK
    worst = [0.0, 0.0, -np.inf]
    for (b, h) in heads:
        q, k, v = (to64(x[n][b, h]) for n in ("q", "k", "v"))
        hm = None if bmask is None else (bmask.numpy() if bmask.dim() == 2 else bmask[b, h].numpy())
        o_ref, lse_ref = oracle.attention_fwd(q, k, v, False, w.scale, rows=rows, window=window, block_mask=hm)
        og = to64(o[b, h]) if rows is None else to64(o[b, h])[rows]
        lg = to64(lse[b, h]) if rows is None else to64(lse[b, h])[rows]
        e_o, e_l, e_ox, dead_ok = fwd_errors(og, lg, o_ref, lse_ref)
        assert dead_ok, f"head {(b, h)}: rows without keys must give O = 0, lse = -inf"
        worst = [max(worst[0], e_o), max(worst[1], e_l), max(worst[2], e_ox)]
    print(f"{w.name} window={window} mask={'none' if bmask is None else tuple(bmask.shape)}: "
          f"max|dO|={worst[0]:.3e} (beyond bf16 rounding {worst[2]:.3e}) max|dlse|={worst[1]:.3e}")
    assert worst[2] <= TOL_O_BF16 and worst[1] <= TOL_LSE, worst


SHAPES = [(1, 2, 700, 700, 128), (1, 2, 300, 900, 64), (1, 2, 900, 300, 256), (2, 1, 520, 520, 64)]
WINDOWS = [(127, 0), (300, 0), (0, 0), (64, 64), (-1, 5), (200, -1)]


@pytest.mark.parametrize("B,H,Tq,Tk,d", SHAPES)
@pytest.mark.parametrize("window", WINDOWS)
def test_windows(fa, B, H, Tq, Tk, d, window):
    w = inputs.small(B, H, Tq, Tk, d, False, seed=Tq + 3 * Tk + d + window[0])
    check(fa, w, window, None, heads_of(w, B * H))


@pytest.mark.parametrize("B,H,Tq,Tk,d", SHAPES)
@pytest.mark.parametrize("per_head", [False, True])
def test_block_masks(fa, B, H, Tq, Tk, d, per_head):
    w = inputs.small(B, H, Tq, Tk, d, False, seed=Tq + 5 * Tk + d)
    bm = random_mask(B, H, Tq, Tk, per_head, seed=Tq + Tk + d)
    check(fa, w, (-1, -1), bm, heads_of(w, B * H))
    check(fa, w, (-1, 0), bm, heads_of(w, B * H))          # block mask inside the causal mask
    check(fa, w, (150, 10), bm, heads_of(w, B * H))        # and inside a window


def test_causal_window_is_fa_fwd(fa):
    w = inputs.small(2, 2, 777, 777, 128, True, seed=9)
    x = inputs.generate(w, with_grad=False, device="cuda")
    o1, l1 = fa.attention_forward(x["q"], x["k"], x["v"], True, w.scale)
    o2, l2 = fa.attention_forward(x["q"], x["k"], x["v"], False, w.scale, window=(-1, 0))
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_sliding_window_4096(fa):
    """The 4096/d128 workload's inputs under a 1024-key causal sliding window."""
    w = inputs.WORKLOADS["fwd_b8h32_t4096_d128_causal"]
    check(fa, w, (1023, 0), None, heads_of(w, 4), rows=rows_of(w.Tq, 512))


def test_masked_errors(fa):
    q = torch.randn(1, 1, 64, 64, device="cuda").to(torch.bfloat16)
    o, lse = torch.empty_like(q), torch.empty(1, 1, 64, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_masked(q, q, q, o, lse, (-2, 0), None, 0.1)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        fa.fa_fwd_masked(q, q, q, o, lse, (-1, 0), torch.ones(2, 2, dtype=torch.uint8, device="cuda"), 0.1)
    assert fa.fa_sync_status() == fa.FA_OK


# ---------------------------------------------------------------- backward under masks
GUARD = 1 << 20
def check_bwd(fa, w, window, bmask, heads, deterministic=False):
    x = inputs.generate(w, with_grad=True, device="cuda")
    bm_dev = None if bmask is None else bmask.to("cuda")
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], False, w.scale, window=window, block_mask=bm_dev)
    # a guard band after the workspace: the kernels must leave it untouched
    need = fa.fa_bwd_workspace_bytes(w.B, w.H, w.Tq, w.Tk, w.d)
    ws = torch.full((need + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    dq, dk, dv = fa.attention_backward(x["q"], x["k"], x["v"], o, lse, x["do"], False, w.scale, workspace=ws[:need],
                                       window=window, block_mask=bm_dev, deterministic=deterministic)
    assert fa.fa_sync_status() == fa.FA_OK
    assert bool(torch.all(ws[need:] == 0xA5)), "write past the end of the workspace"
    worst = {"dq": 0.0, "dk": 0.0, "dv": 0.0}
    for (b, h) in heads:
        q, k, v, do = (to64(x[n][b, h]) for n in ("q", "k", "v", "do"))
        hm = None if bmask is None else (bmask.numpy() if bmask.dim() == 2 else bmask[b, h].numpy())
        ref = oracle.attention_bwd(q, k, v, do, False, w.scale, window=window, block_mask=hm)
        for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            g = to64(t[b, h])
            assert np.all(np.isfinite(g)), n
            worst[n] = max(worst[n], float((np.abs(g - ref[n]) - half_ulp_bf16(ref[n])).max()))
    print(f"{w.name} bwd window={window} mask={'none' if bmask is None else tuple(bmask.shape)} "
          f"det={deterministic}: beyond bf16 rounding " + " ".join(f"{n}={v:.3e}" for n, v in worst.items()))
    for n, v in worst.items():
        assert v <= TOL_GRAD, (n, worst)
    return dq, dk, dv


BWD_SHAPES = [(1, 2, 700, 700, 128), (1, 2, 300, 900, 64), (1, 2, 900, 300, 128), (2, 1, 520, 520, 64)]


@pytest.mark.parametrize("B,H,Tq,Tk,d", BWD_SHAPES)
@pytest.mark.parametrize("window", [(127, 0), (0, 0), (64, 64), (-1, 5), (200, -1)])
def test_bwd_windows(fa, B, H, Tq, Tk, d, window):
    w = inputs.small(B, H, Tq, Tk, d, False, seed=Tq + 3 * Tk + d + window[0], backward=True)
    check_bwd(fa, w, window, None, heads_of(w, B * H))


@pytest.mark.parametrize("B,H,Tq,Tk,d", BWD_SHAPES)
@pytest.mark.parametrize("per_head", [False, True])
def test_bwd_block_masks(fa, B, H, Tq, Tk, d, per_head):
    w = inputs.small(B, H, Tq, Tk, d, False, seed=Tq + 5 * Tk + d, backward=True)
    bm = random_mask(B, H, Tq, Tk, per_head, seed=Tq + Tk + d)
    check_bwd(fa, w, (-1, -1), bm, heads_of(w, B * H))
    check_bwd(fa, w, (150, 10), bm, heads_of(w, B * H))


def test_bwd_masked_deterministic(fa):
    w = inputs.small(1, 2, 700, 700, 128, False, seed=21, backward=True)
    bm = random_mask(1, 2, 700, 700, True, seed=22)
    a = check_bwd(fa, w, (300, 0), bm, heads_of(w, 2), deterministic=True)
    b = check_bwd(fa, w, (300, 0), bm, heads_of(w, 2), deterministic=True)
    assert all(torch.equal(s.view(torch.int16), t.view(torch.int16)) for s, t in zip(a, b))
