"""FP8 forward of the method, fp64 reference -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the product path never does.

atlas.blal.pro "FlashAttention -- IO-Aware Exact Attention", "The version ladder:
FA1 -> FA2 -> FA3" (the FA3 entry) names the FP8 forward's two devices: block
quantization (one scale per block of rows) and incoherent processing (a random
rotation applied to Q and K before quantizing, which spreads outlier features over
all channels while leaving Q K^T unchanged).  "Honest caveats & open questions"
adds that the result is a precision trade-off, so the quantities here define what
the FP8 path computes and its error budget is derived from them.

Readings (the pages fix none of these details):
  * format: e4m3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
    infinities, largest finite 448), round to nearest even, saturating at +-448;
  * rotation: x -> x diag(s) H / sqrt(d), s a vector of d random signs (an input),
    H the d x d Sylvester Hadamard matrix; applied to Q and K only;
  * blocks: one scale per 128 rows of Q and per 128 keys of K (the tile height of
    the forward), chosen so that the block's largest |value| maps to 448; V gets one
    scale per feature channel over all keys of a head, which factors out of P V;
  * the decision of each code is taken in fp32, as the kernel takes it: the
    Hadamard sums with the butterfly order below, the reciprocal 448 / amax and the
    product x * (448 / amax), each rounded to fp32, then rounded to e4m3.
The exact FP8 result is then plain attention (the fp64 oracle) over the
dequantized values q8 * sq, k8 * sk, v8 * sv.
"""
from __future__ import annotations

import numpy as np

from . import attention_fwd

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value (ties to even), saturating at +-448: the binade of |x| is
    [2^e, 2^(e+1)) with e >= -6 (below 2^-6 the subnormal spacing 2^-9 holds), and the
    grid step inside it is 2^(e-3).  fp64 in and out."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, ex = np.frexp(ax)                         # ax = m 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6)
    step = np.ldexp(1.0, e - 3)
    q = np.round(ax / step) * step               # ax / step is exact; numpy rounds half to even
    return np.copysign(np.minimum(q, E4M3_MAX), x)


def fwht_f32(x) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform along the last axis, in fp32: for
    h = 1, 2, 4, ..., d/2 each pair (i, i + h) with i & h = 0 becomes (a + b, a - b),
    every sum rounded to fp32.  Equals x @ H (Sylvester order) up to that rounding."""
    y = np.array(x, dtype=np.float32)
    d = y.shape[-1]
    assert d & (d - 1) == 0, "d must be a power of two"
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(*lead, d // (2 * h), 2, h)
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(*lead, d)
        h *= 2
    return y


def _codes(vals32: np.ndarray, amax32: np.float32) -> np.ndarray:
    """e4m3 codes (as fp64 values) of fp32 values under the scale that maps amax to 448."""
    if amax32 > 0:
        inv = np.float32(E4M3_MAX) / amax32                  # fp32 division, rounded once
        return e4m3_round((vals32 * inv).astype(np.float32))  # fp32 product, rounded once
    return np.zeros(vals32.shape)


def quantize_rows(x, signs=None, block: int = BLOCK):
    """Block quantization of a (T, d) operand (Q or K of one head).  With `signs` the
    rows are rotated first (incoherent processing).  Returns (codes (T, d) as fp64 e4m3
    values, descale (ceil(T/block),) fp64) with x diag(s) H / sqrt(d) ~= codes * descale
    (per row block), or x ~= codes * descale without rotation."""
    x = np.asarray(x, dtype=np.float64)
    T, d = x.shape
    y = fwht_f32(x * np.asarray(signs, dtype=np.float64)) if signs is not None else x.astype(np.float32)
    nb = -(-T // block)
    codes = np.zeros((T, d))
    descale = np.zeros(nb)
    for b in range(nb):
        blk = y[b * block:(b + 1) * block]
        amax = np.float32(np.abs(blk).max()) if blk.size else np.float32(0)
        codes[b * block:(b + 1) * block] = _codes(blk, amax)
        descale[b] = float(amax) / E4M3_MAX / (np.sqrt(d) if signs is not None else 1.0)
    return codes, descale


def quantize_channels(v):
    """Per-channel quantization of V (Tk, d): channel c is scaled so that its largest
    |value| over all keys maps to 448.  Returns (codes (Tk, d), descale (d,))."""
    v32 = np.asarray(v, dtype=np.float32)
    Tk, d = v32.shape
    codes = np.zeros((Tk, d))
    descale = np.zeros(d)
    for c in range(d):
        amax = np.float32(np.abs(v32[:, c]).max()) if Tk else np.float32(0)
        codes[:, c] = _codes(v32[:, c], amax)
        descale[c] = float(amax) / E4M3_MAX
    return codes, descale


def dequantized(q, k, v, signs=None, block: int = BLOCK):
    """The FP8 operands as the attention sees them: (q^, k^, v^) in fp64."""
    q8, sq = quantize_rows(q, signs, block)
    k8, sk = quantize_rows(k, signs, block)
    v8, sv = quantize_channels(v)
    return (q8 * np.repeat(sq, block)[:q8.shape[0], None], k8 * np.repeat(sk, block)[:k8.shape[0], None],
            v8 * sv[None, :])


def attention_fwd_fp8(q, k, v, causal: bool, scale: float, signs=None, rows=None, nthreads=None):
    """Exact attention over the dequantized FP8 operands: (O, lse) in fp64."""
    qh, kh, vh = dequantized(q, k, v, signs)
    return attention_fwd(qh, kh, vh, causal, scale, rows=rows, nthreads=nthreads)
