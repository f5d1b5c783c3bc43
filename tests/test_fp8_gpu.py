"""FP8 forward (fa_fp8_quantize + fa_fwd_fp8) against the FP8 oracle (oracle/fp8.py).

atlas.blal.pro "FlashAttention -- IO-Aware Exact Attention", "The version ladder" (the FA3
entry: block quantization and incoherent processing) and "Honest caveats & open questions"
(FP8 is a precision trade-off, so its error budget is its own).

* Quantization: the e4m3 codes are integer decisions taken in fp32 on both sides, so they
  must match the oracle's bit for bit; the descales to fp32 rounding.
* Forward: the oracle is exact attention over the dequantized operands.  The kernel
  differs from it by rounding P~ to e4m3 before the P V product (scores, row sums and O
  stay fp32) and by the bf16 output.  Each probability p_l is rounded with relative error
  at most 2^-4, or absolute 2^-14 in units of the row's largest weight when it is
  subnormal in e4m3, so per element
      |O - O_ref| <= 2^-4 sum_l p_l |v_l| + 2^-14 sum_l |v_l| / L + ulp_bf16 / 2 + 1e-4,
  L = sum_l exp(s_l - max s) >= 1; every element is held to that.  The bound is loose
  (the roundings are independent); the RMS error is also held to twice the RMS that
  independent uniform roundings predict, which a wrong scale or a lost tile exceeds.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
from exact_io_aware_05_gb300 import inputs
from gpu_util import half_ulp_bf16, heads_of, rows_of, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_io_aware_05_gb300 import fa as _fa
    return _fa


def e4m3_values(codes: torch.Tensor) -> np.ndarray:
    return codes.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def signs_for(d, seed):
    return inputs.rotation_signs(d, seed)


# ---------------------------------------------------------------- quantization
QSHAPES = [(1, 2, 300, 200, 64), (2, 1, 128, 130, 128), (1, 2, 257, 700, 128), (1, 1, 90, 33, 256)]


@pytest.mark.parametrize("B,H,Tq,Tk,d", QSHAPES)
@pytest.mark.parametrize("rotate", [False, True])
def test_quantize_matches_oracle(fa, B, H, Tq, Tk, d, rotate):
    w = inputs.small(B, H, Tq, Tk, d, False, seed=Tq + 7 * Tk + d)
    x = inputs.generate(w, with_grad=False, device="cuda")
    s = signs_for(d, 11) if rotate else None
    out = fa.fa_fp8_quantize(x["q"], x["k"], x["v"], None if s is None else s.cuda())
    torch.cuda.synchronize()
    assert fa.fa_sync_status() == fa.FA_OK
    sn = None if s is None else s.double().numpy()
    ld = fa.fa_fp8_vt_stride(Tk)
    assert ld % 16 == 0 and ld >= Tk
    for b in range(B):
        for h in range(H):
            q, k, v = (to64(x[n][b, h]) for n in ("q", "k", "v"))
            for name, src, T in (("q", q, Tq), ("k", k, Tk)):
                codes, ds = ofp8.quantize_rows(src, sn)
                got = e4m3_values(out[name + "8"][b, h])
                assert np.array_equal(got, codes), f"{name} codes differ at {np.argwhere(got != codes)[:5]}"
                gds = out[name + "_descale"][b, h].cpu().double().numpy()
                assert np.allclose(gds, ds, rtol=1e-6, atol=0), name
            codes, ds = ofp8.quantize_channels(v)
            got = e4m3_values(out["vt8"][b, h][:, :Tk]).T
            assert np.array_equal(got, codes), "v codes"
            assert np.allclose(out["v_descale"][b, h].cpu().double().numpy(), ds, rtol=1e-6, atol=0)


# ---------------------------------------------------------------- forward
def fwd_bound(qh, kh, vh, causal, scale, rows=None):
    """Per-element bound and predicted variance of the kernel's P rounding (see module doc)."""
    Tq, Tk = qh.shape[0], kh.shape[0]
    r = np.arange(Tq) if rows is None else np.asarray(rows)
    s = scale * qh[r] @ kh.T
    if causal:
        allowed = np.arange(Tk)[None, :] <= (r[:, None] + Tk - Tq)
        s = np.where(allowed, s, -np.inf)
    mx = s.max(axis=1, keepdims=True)
    live = np.isfinite(mx[:, 0])
    e = np.where(live[:, None], np.exp(s - np.where(live[:, None], mx, 0)), 0.0)
    L = e.sum(axis=1, keepdims=True)
    p = e / np.where(L > 0, L, 1)
    av = np.abs(vh)
    bound = 2.0 ** -4 * (p @ av) + 2.0 ** -14 * ((e > 0) @ av) / np.where(L > 0, L, 1)
    var = (2.0 ** -8 * 0.18) * ((p ** 2) @ (vh ** 2))
    return bound, var


def check_fwd(fa, w, signs_seed, heads, rows=None, outliers=None):
    x = inputs.generate(w, with_grad=False, device="cuda")
    if outliers is not None:
        for n in ("q", "k"):
            x[n][..., outliers] *= 20.0
    s = None if signs_seed is None else signs_for(w.d, signs_seed)
    o, lse, _ = fa.attention_forward_fp8(x["q"], x["k"], x["v"], w.causal, w.scale,
                                         signs=None if s is None else s.cuda())
    torch.cuda.synchronize()
    assert fa.fa_sync_status() == fa.FA_OK
    sn = None if s is None else s.double().numpy()
    err2 = var2 = 0.0
    n_el = 0
    worst = 0.0
    for (b, h) in heads:
        q, k, v = (to64(x[n][b, h]) for n in ("q", "k", "v"))
        qh, kh, vh = ofp8.dequantized(q, k, v, sn)
        o_ref, lse_ref = oracle.attention_fwd(qh, kh, vh, w.causal, w.scale, rows=rows)
        og = to64(o[b, h]) if rows is None else to64(o[b, h])[rows]
        lg = to64(lse[b, h]) if rows is None else to64(lse[b, h])[rows]
        live = np.isfinite(lse_ref)
        assert np.all(og[~live] == 0) and np.all(np.isinf(lg[~live]))
        bound, var = fwd_bound(qh, kh, vh, w.causal, w.scale, rows)
        err = np.abs(og - o_ref)
        tol = bound + half_ulp_bf16(o_ref) + 1e-4
        worst = max(worst, float((err / tol).max()))
        assert np.all(err <= tol), f"head {(b, h)}: {np.argwhere(err > tol)[:5]}"
        assert np.abs(lg[live] - lse_ref[live]).max() <= 1e-4
        err2 += float((err ** 2).sum())
        var2 += float((var + half_ulp_bf16(o_ref) ** 2 / 3).sum())
        n_el += err.size
    ratio = np.sqrt(err2 / max(var2, 1e-300))
    print(f"{w.name} fp8 signs={signs_seed}: rms error {np.sqrt(err2 / n_el):.3e}, "
          f"predicted {np.sqrt(var2 / n_el):.3e} (ratio {ratio:.2f}), worst element at {worst:.2f} of its bound")
    assert ratio <= 2.0
    return np.sqrt(err2 / n_el)


FSHAPES = [(1, 2, 700, 700, True), (1, 2, 700, 700, False), (2, 1, 300, 900, True), (1, 2, 900, 300, True),
           (1, 1, 128, 128, False), (1, 2, 1, 77, True), (1, 1, 520, 1000, False)]


@pytest.mark.parametrize("B,H,Tq,Tk,causal", FSHAPES)
@pytest.mark.parametrize("signs_seed", [None, 5])
def test_fwd_fp8_small(fa, B, H, Tq, Tk, causal, signs_seed):
    w = inputs.small(B, H, Tq, Tk, 128, causal, seed=3 * Tq + Tk + int(causal))
    check_fwd(fa, w, signs_seed, heads_of(w, B * H))


def test_fwd_fp8_workload(fa):
    """The 4096/d128 causal shape with the rotation: sampled heads and rows."""
    w = inputs.WORKLOADS["fwd_fp8_b8h32_t4096_d128_causal"]
    check_fwd(fa, w, 1, heads_of(w, 4), rows=rows_of(w.Tq, 384))


def test_rotation_lowers_gpu_error(fa):
    """With outlier channels in Q and K, the rotated FP8 forward is closer to exact bf16
    attention than the unrotated one."""
    w = inputs.small(1, 2, 1024, 1024, 128, False, seed=77, scale=1.0 / 128)
    out = [3, 40, 77, 100]
    x = inputs.generate(w, with_grad=False, device="cuda")
    for n in ("q", "k"):
        x[n][..., out] *= 20.0
    errs = []
    for s in (None, signs_for(128, 5).cuda()):
        o, _, _ = fa.attention_forward_fp8(x["q"], x["k"], x["v"], False, w.scale, signs=s)
        torch.cuda.synchronize()
        e = 0.0
        for h in range(2):
            q, k, v = (to64(x[n][0, h]) for n in ("q", "k", "v"))
            o_ref, _ = oracle.attention_fwd(q, k, v, False, w.scale)
            e += float(((to64(o[0, h]) - o_ref) ** 2).mean())
        errs.append(np.sqrt(e / 2))
    print(f"rms error against exact attention: no rotation {errs[0]:.3e}, rotation {errs[1]:.3e}")
    assert errs[1] * 1.5 <= errs[0]


def test_fp8_errors(fa):
    dev = "cuda"
    q = torch.randn(1, 1, 64, 64, device=dev).to(torch.bfloat16)
    x = fa.fa_fp8_quantize(q, q, q)
    o, lse = torch.empty_like(q), torch.empty(1, 1, 64, device=dev)
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_fp8(x, o, lse, False, 0.1)                 # d = 64: forward is d = 128 only
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    q = torch.randn(1, 1, 64, 128, device=dev).to(torch.bfloat16)
    x = fa.fa_fp8_quantize(q, q, q)
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_fp8(x, torch.empty_like(q), lse, False, float("nan"))
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    k0 = torch.empty(1, 1, 0, 128, device=dev, dtype=torch.bfloat16)
    o, lse, _ = fa.attention_forward_fp8(q, k0, k0, False, 0.1)  # no keys: O = 0, lse = -inf
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isinf(lse))
    assert fa.fa_sync_status() == fa.FA_OK
