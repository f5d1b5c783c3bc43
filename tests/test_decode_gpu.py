"""Split-KV decode (fa_decode) against the fp64 oracle: the same O and lse as the
forward pass for a few query rows per head (atlas.blal.pro "FlashAttention --
IO-Aware Exact Attention", "Honest caveats & open questions": FlashDecoding splits
the keys; the chunks are merged by the online-softmax rescale of zerotofrontier.app
"FlashAttention", "The forward pass").  Every element for small and ragged shapes
(chunk and tile edges, causal rows without keys), sampled heads at the two decode
workloads, and the host-side errors."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_05_gb300 import inputs
from gpu_util import TOL_LSE, TOL_O_BF16, fwd_errors, heads_of, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_io_aware_05_gb300 import fa as _fa
    return _fa


def check(fa, w, heads):
    x = inputs.generate(w, with_grad=False, device="cuda")
    o, lse = fa.attention_decode(x["q"], x["k"], x["v"], w.causal, w.scale)
    assert fa.fa_sync_status() == fa.FA_OK
    worst = [0.0, 0.0, -np.inf]
    for (b, h) in heads:
        q, k, v = (to64(x[n][b, h]) for n in ("q", "k", "v"))
        o_ref, lse_ref = oracle.attention_fwd(q, k, v, w.causal, w.scale)
        e_o, e_l, e_ox, dead_ok = fwd_errors(to64(o[b, h]), to64(lse[b, h]), o_ref, lse_ref)
        assert dead_ok, f"head {(b, h)}: rows without keys must give O = 0, lse = -inf"
        worst = [max(worst[0], e_o), max(worst[1], e_l), max(worst[2], e_ox)]
    print(f"{w.name}: max|dO|={worst[0]:.3e} (beyond bf16 output rounding {worst[2]:.3e}) max|dlse|={worst[1]:.3e}")
    assert worst[2] <= TOL_O_BF16 and worst[1] <= TOL_LSE, worst
    return o, lse


SMALL = [
    # B, H, Tq, Tk, d, causal: tile (32) and chunk edges, Tq > Tk (rows without keys)
    (1, 2, 1, 1, 128, True), (1, 2, 1, 31, 128, False), (1, 2, 1, 33, 64, True), (2, 3, 1, 1000, 128, True),
    (1, 2, 3, 4097, 128, True), (1, 2, 16, 777, 64, False), (1, 1, 16, 10, 128, True), (1, 2, 5, 3, 64, True),
    (1, 2, 8, 2500, 256, True), (1, 2, 2, 300, 256, False), (3, 1, 4, 20000, 64, False),
]


@pytest.mark.parametrize("B,H,Tq,Tk,d,causal", SMALL)
def test_decode_small(fa, B, H, Tq, Tk, d, causal):
    w = inputs.small(B, H, Tq, Tk, d, causal, seed=13 * Tk + Tq + d)
    check(fa, w, heads_of(w, B * H))


@pytest.mark.parametrize("name", ["decode_b8h32_q1_k32768_d128", "decode_b1h32_q4_k131072_d128"])
def test_decode_workloads(fa, name):
    w = inputs.WORKLOADS[name]
    check(fa, w, heads_of(w, 6))


def test_decode_matches_forward(fa):
    """The split and the single-pass kernels compute the same quantity: at one query row,
    their outputs agree to bf16 rounding."""
    w = inputs.small(2, 4, 1, 9000, 128, True, seed=3)
    x = inputs.generate(w, with_grad=False, device="cuda")
    o1, l1 = fa.attention_decode(x["q"], x["k"], x["v"], True, w.scale)
    o2, l2 = fa.attention_forward(x["q"], x["k"], x["v"], True, w.scale)
    torch.cuda.synchronize()
    assert float((o1.float() - o2.float()).abs().max()) <= 2e-2
    assert float((l1 - l2).abs().max()) <= 1e-4


def test_decode_edges(fa):
    dev = "cuda"
    q = torch.randn(1, 2, 3, 64, device=dev).to(torch.bfloat16)
    k0 = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    o, lse = fa.attention_decode(q, k0, k0, False, 0.125)       # no key at all
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isinf(lse)) and torch.all(lse < 0)
    q17 = torch.randn(1, 1, 17, 128, device=dev).to(torch.bfloat16)
    k = torch.randn(1, 1, 64, 128, device=dev).to(torch.bfloat16)
    assert fa.fa_decode_workspace_bytes(1, 1, 17, 64, 128) == 0
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FAError) as e:
        fa.fa_decode(q17, k, k, torch.empty_like(q17), torch.empty(1, 1, 17, device=dev), False, 0.1, ws)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    q1 = torch.randn(1, 1, 1, 128, device=dev).to(torch.bfloat16)
    small = torch.empty(16, dtype=torch.uint8, device=dev)
    kk = torch.randn(1, 1, 4096, 128, device=dev).to(torch.bfloat16)
    with pytest.raises(fa.FAError) as e:
        fa.fa_decode(q1, kk, kk, torch.empty_like(q1), torch.empty(1, 1, 1, device=dev), False, 0.1, small)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    assert fa.fa_sync_status() == fa.FA_OK
