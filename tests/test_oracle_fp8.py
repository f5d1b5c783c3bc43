"""Pins of the FP8 oracle (oracle/fp8.py), each against something other than its own
formula: torch's float8_e4m3fn cast, scipy's Hadamard matrix, an enumeration of the
256 e4m3 codes, the invariance of Q K^T under the rotation, special cases that reduce
to the plain oracle, and the pages' claim that incoherent processing lowers the FP8
error (atlas.blal.pro "FlashAttention -- IO-Aware Exact Attention", "The version
ladder: FA1 -> FA2 -> FA3": FA3's FP8 error is 2.6x below a naive FP8 baseline)."""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from oracle import fp8


def e4m3_grid() -> np.ndarray:
    """Every finite e4m3 value, from the 256 bit patterns decoded by torch."""
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return np.unique(codes[np.isfinite(codes)])


def test_e4m3_grid_fixed_points_and_extremes():
    g = e4m3_grid()
    assert g.size == 253 and g.max() == 448.0 and g[g > 0].min() == 2.0 ** -9   # +-0 merge, 2 NaNs
    assert np.array_equal(fp8.e4m3_round(g), g)
    assert fp8.e4m3_round(1e6) == 448.0 and fp8.e4m3_round(-470.0) == -448.0      # saturation


def test_e4m3_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        np.sign(rng.standard_normal(20000)) * np.exp2(rng.uniform(-12, np.log2(464), 20000)),
        rng.standard_normal(5000) * 50,
    ])
    x = x[np.abs(x) <= 464]
    g = e4m3_grid()
    mids = (g[1:] + g[:-1]) / 2                               # ties: torch rounds to even
    x = np.concatenate([x, mids[np.abs(mids) <= 464]])
    ref = torch.tensor(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(fp8.e4m3_round(x), ref)


@pytest.mark.parametrize("d", [2, 8, 64, 128, 256])
def test_fwht_is_sylvester_hadamard(d):
    rng = np.random.default_rng(d)
    H = scipy.linalg.hadamard(d).astype(np.float64)
    xi = rng.integers(-50, 50, size=(7, d)).astype(np.float64)   # exact in fp32
    assert np.array_equal(fp8.fwht_f32(xi).astype(np.float64), xi @ H)
    x = rng.standard_normal((9, d))
    y = fp8.fwht_f32(x).astype(np.float64)
    bound = np.log2(d) * 2.0 ** -23 * (np.abs(x) @ np.abs(H))
    assert np.all(np.abs(y - x @ H) <= bound + 1e-30)
    assert np.allclose(fp8.fwht_f32(y) / d, x.astype(np.float32), atol=1e-5)   # H H = d I


def test_rotation_keeps_scores():
    rng = np.random.default_rng(1)
    d = 128
    s = rng.choice([-1.0, 1.0], size=d)
    q, k = rng.standard_normal((20, d)), rng.standard_normal((30, d))
    qr = fp8.fwht_f32(q * s).astype(np.float64) / np.sqrt(d)
    kr = fp8.fwht_f32(k * s).astype(np.float64) / np.sqrt(d)
    assert np.allclose(qr @ kr.T, q @ k.T, atol=2e-4)


def test_quantize_rows_blocks():
    rng = np.random.default_rng(2)
    T, d = 300, 64
    x = rng.standard_normal((T, d)) * np.exp2(rng.integers(-3, 4, size=(T, 1)))
    x[256:] = 0.0                                      # an all-zero last block
    s = rng.choice([-1.0, 1.0], size=d)
    g = e4m3_grid()
    for signs in (None, s):
        codes, ds = fp8.quantize_rows(x, signs)
        assert codes.shape == (T, d) and ds.shape == (3,)
        assert np.array_equal(fp8.e4m3_round(codes), codes)          # on the grid
        assert np.abs(codes[:128]).max() == 448.0 and np.abs(codes[128:256]).max() == 448.0
        assert np.all(codes[256:] == 0) and ds[2] == 0
        xr = x if signs is None else fp8.fwht_f32(x * signs).astype(np.float64) / np.sqrt(d)
        for b in range(2):
            blk, cb = xr[b * 128:(b + 1) * 128], codes[b * 128:(b + 1) * 128]
            # each code is the grid value nearest to the scaled input (brute force over the grid)
            t = blk / ds[b]
            nearest = g[np.abs(t[..., None] - g).argmin(axis=-1)]
            close = np.abs(np.abs(t - nearest) - np.abs(t - cb)) <= 1e-5 * np.abs(t)
            assert np.all(close)
            # dequantization error within half a grid step (relative 2^-4, or 2^-10 absolute)
            err = np.abs(cb * ds[b] - blk)
            assert np.all(err <= (np.maximum(np.abs(blk) / 16, 2.0 ** -10 * ds[b])) * (1 + 1e-5))


def test_quantize_channels():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((500, 32)) * np.exp2(rng.integers(-4, 5, size=(1, 32)))
    codes, ds = fp8.quantize_channels(v)
    assert np.all(np.abs(codes).max(axis=0) == 448.0)
    assert np.all(np.abs(codes * ds - v) <= np.maximum(np.abs(v) / 16, 2.0 ** -10 * ds) * (1 + 1e-5))


def test_exactly_representable_inputs_reduce_to_the_plain_oracle():
    """Without rotation, inputs that are e4m3 values whose block maximum is 448 times a
    power of two quantize without error: the FP8 result is then the plain result."""
    rng = np.random.default_rng(4)
    g = e4m3_grid()
    T, d = 200, 16

    def draw(n):
        """two row blocks with different scales, each holding +-448 times its scale"""
        x = rng.choice(g[np.abs(g) <= 448], size=(n, d))
        x[0, 0] = 448.0
        x[128, 0] = -448.0
        x[:128] *= 2.0 ** -6
        x[128:] *= 2.0 ** -9
        return x

    q, k = draw(T), draw(T)
    v = rng.choice(g[np.abs(g) <= 448], size=(T, d))
    v[3, :] = 448.0
    v *= 2.0 ** -5
    for causal in (False, True):
        o1, l1 = oracle.attention_fwd(q, k, v, causal, 0.3)
        o2, l2 = fp8.attention_fwd_fp8(q, k, v, causal, 0.3)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_incoherent_processing_lowers_the_error():
    """Inputs with a few outlier channels (the case the rotation is for): the RMS error
    of O against exact attention with per-block scales and the rotation is well below
    that of a naive FP8 baseline (one scale for the whole head, no rotation)."""
    rng = np.random.default_rng(5)
    T, d = 512, 128
    q, k, v = (rng.standard_normal((T, d)) for _ in range(3))
    out = rng.choice(d, size=4, replace=False)
    q[:, out] *= 20.0
    k[:, out] *= 20.0
    scale = 1.0 / np.sqrt(d) / 8
    s = rng.choice([-1.0, 1.0], size=d)
    o_ref, _ = oracle.attention_fwd(q, k, v, False, scale)
    o_fp8, _ = fp8.attention_fwd_fp8(q, k, v, False, scale, signs=s)
    qn, _ = fp8.quantize_rows(q, None, block=T)
    kn, _ = fp8.quantize_rows(k, None, block=T)
    qd = qn * np.abs(q).max() / 448
    kd = kn * np.abs(k).max() / 448
    vn, vs = fp8.quantize_rows(v, None, block=T)
    o_naive, _ = oracle.attention_fwd(qd, kd, vn * vs[0], False, scale)
    e_fp8 = np.sqrt(np.mean((o_fp8 - o_ref) ** 2))
    e_naive = np.sqrt(np.mean((o_naive - o_ref) ** 2))
    print(f"rms error: block + rotation {e_fp8:.3e}, naive {e_naive:.3e}, ratio {e_naive / e_fp8:.2f}")
    assert e_naive / e_fp8 >= 2.0
