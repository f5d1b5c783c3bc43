"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and the
oracle on the same seeded inputs, and measure element-wise errors."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from exact_io_aware_05_gb300 import inputs

# Tolerances stated for the path: bf16 inputs with fp32 accumulation
TOL_O_BF16 = 1e-2
TOL_LSE = 1e-4
TOL_GRAD = 2e-2
TOL_O_F32 = 1e-5


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even to bf16 (for reporting output quantisation)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()


def heads_of(w: inputs.Workload, n: int, seed: int = 0):
    """n (b, h) pairs including the first and the last head."""
    all_h = [(b, h) for b in range(w.B) for h in range(w.H)]
    if n >= len(all_h):
        return all_h
    if n < 2:
        return all_h[:n]
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, len(all_h) - 1), size=n - 2, replace=False)
    return [all_h[0]] + [all_h[i] for i in sorted(mid)] + [all_h[-1]]


def rows_of(T: int, n: int, block: int = 128, seed: int = 0):
    """Sampled query rows: 0, T-1, block edges and random rows."""
    rng = np.random.default_rng(seed)
    fixed = {0, T - 1}
    for e in range(block, T, block * max(1, (T // block) // 16)):
        fixed.update({e - 1, e})
    fixed = sorted(r for r in fixed if 0 <= r < T)
    rest = rng.choice(T, size=max(0, n - len(fixed)), replace=False)
    return np.unique(np.concatenate([np.array(fixed, dtype=np.int64), rest.astype(np.int64)]))


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half a unit in the last place of bf16 at |x| (8 significant bits): the rounding error
    that storing an exact value in a bf16 output alone can cause."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def excess_over_output_rounding(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max of |gpu - ref| - half_ulp_bf16(ref): the error of the computation itself, once the
    unavoidable rounding of an exact result to the bf16 output format is set aside."""
    if ref.size == 0:
        return 0.0
    return float((np.abs(gpu - ref) - half_ulp_bf16(ref)).max())


def fwd_errors(o_gpu, lse_gpu, o_ref, lse_ref):
    """max |O - O_ref|, max |lse - lse_ref| over live rows, the O error in excess of the bf16
    output rounding, and whether the dead (-inf) rows agree."""
    live = np.isfinite(lse_ref)
    dead_ok = bool(np.all(~np.isfinite(lse_gpu[~live])) and np.all(o_gpu[~live] == 0))
    e_o = float(np.abs(o_gpu - o_ref).max()) if o_ref.size else 0.0
    e_o_x = excess_over_output_rounding(o_gpu, o_ref)
    e_l = float(np.abs(lse_gpu[live] - lse_ref[live]).max()) if live.any() else 0.0
    return e_o, e_l, e_o_x, dead_ok


def check_grads(w, x, grads, heads, rows=None, keys=None, tol=TOL_GRAD):
    """Every gradient element within tol of the oracle, beyond half a bf16 ulp of the exact
    value (the rounding of the bf16 output itself)."""
    dq, dk, dv = grads
    worst = {"dq": 0.0, "dk": 0.0, "dv": 0.0}
    raw = dict(worst)
    for (b, h) in heads:
        q, k, v, do = (to64(x[n][b, h]) for n in ("q", "k", "v", "do"))
        ref = oracle.attention_bwd(q, k, v, do, w.causal, w.scale, rows=rows, keys=keys)
        pick = {"dq": (dq, rows), "dk": (dk, keys), "dv": (dv, keys)}
        for n, (t, ix) in pick.items():
            g = to64(t[b, h]) if ix is None else to64(t[b, h])[ix]
            assert np.all(np.isfinite(g)), n
            raw[n] = max(raw[n], float(np.abs(g - ref[n]).max()) if g.size else 0.0)
            worst[n] = max(worst[n], excess_over_output_rounding(g, ref[n]))
    print(f"{w.name}: max|err| " + " ".join(f"{n}={raw[n]:.3e}" for n in raw) +
          " | beyond bf16 output rounding " + " ".join(f"{n}={worst[n]:.3e}" for n in worst))
    for n in worst:
        assert worst[n] <= tol, (n, worst, raw)
    return raw, worst


def assert_same_up_to_add_order(got: torch.Tensor, want: torch.Tensor, what: str = "dq") -> None:
    """Two bf16 results of the same fp32 sums added in different orders (the dQ reduce-adds
    land in whatever order the thread blocks reach them): each element within one bf16 ulp of
    the larger magnitude, plus 1e-5 of the tensor's largest magnitude for fp32 partial sums
    that cancel near zero."""
    a = got.detach().float().cpu().double().numpy()
    b = want.detach().float().cpu().double().numpy()
    m = np.maximum(np.abs(a), np.abs(b))
    ulp = np.where(m > 0, np.exp2(np.floor(np.log2(np.where(m > 0, m, 1.0))) - 7), 0.0)
    floor = 1e-5 * float(np.abs(b).max()) if b.size else 0.0
    bad = np.abs(a - b) > ulp + floor
    assert not bad.any(), (what, int(bad.sum()), float(np.abs(a - b).max()))
