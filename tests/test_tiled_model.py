"""The fp64 tiled model against the naive oracle, and the pages' printed IO counts.

zerotofrontier "FlashAttention" (12.3) says the tiled NumPy forward and
backward agree with naive attention to about 1e-15, prints the traffic of one
run (1.18 million values against 4.46 million, n_r = 8) and the causal tile
count (72 of 128).  The run's T, d, B_r, B_c are reconstructed in
tests/golden/io_counts.json.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import tiled

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(Tq, Tk, d, seed, dO=False):
    r = np.random.default_rng(seed)
    out = [r.normal(size=(Tq, d)), r.normal(size=(Tk, d)), r.normal(size=(Tk, d))]
    if dO:
        out.append(r.normal(size=(Tq, d)))
    return out


CASES = [(40, 40, 16, 16, False), (40, 40, 16, 8, True), (37, 53, 8, 24, True), (53, 37, 24, 8, True),
         (70, 70, 32, 16, True), (29, 45, 16, 16, False), (256, 256, 128, 64, True)]


@pytest.mark.parametrize("Tq,Tk,Br,Bc,causal", CASES)
def test_tiled_forward_equals_naive(Tq, Tk, Br, Bc, causal):
    q, k, v = _inputs(Tq, Tk, 8, seed=Tq * 7 + Tk)
    res = tiled.flash_forward(q, k, v, Br, Bc, causal=causal, scale=0.37)
    o, lse = oracle.attention_fwd(q, k, v, causal, 0.37)
    live = np.isfinite(lse)
    assert np.array_equal(np.isfinite(res.lse), live)
    np.testing.assert_allclose(res.o, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(res.lse[live], lse[live], rtol=0, atol=1e-12)


@pytest.mark.parametrize("Tq,Tk,Br,Bc,causal", CASES)
def test_tiled_backward_equals_naive(Tq, Tk, Br, Bc, causal):
    q, k, v, dO = _inputs(Tq, Tk, 8, seed=Tq * 5 + Tk, dO=True)
    g = oracle.attention_bwd(q, k, v, dO, causal, 0.37, want_o=True)
    dq, dk, dv, _ = tiled.flash_backward(q, k, v, g["o"], dO, g["lse"], Br, Bc, causal, 0.37)
    for a, b in ((dq, g["dq"]), (dk, g["dk"]), (dv, g["dv"])):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_first_with_first_skip_drops_keys():
    """Comparing the first key with the FIRST query of a block (the off-by-one the page
    warns about) skips tiles that some rows need; the last-query test keeps them."""
    T, Br, Bc = 64, 32, 16
    wrong = sum(1 for i in range(T // Br) for j in range(T // Bc) if not j * Bc > i * Br)
    right = tiled.causal_tiles_visited(T, Br, Bc)
    assert wrong < right


def test_printed_io_counts():
    g = json.load(open(os.path.join(GOLD, "io_counts.json")))
    rc, pr = g["reconstructed"], g["printed"]
    T, d, Br, Bc = rc["T"], rc["d"], rc["Br"], rc["Bc"]
    q, k, v = _inputs(T, T, d, seed=11)
    res = tiled.flash_forward(q, k, v, Br, Bc)
    assert math.ceil(T / Br) == pr["n_r"]
    assert res.counter.total == tiled.fa2_order_accesses(T, d, Br) == 1_180_672
    assert round(res.counter.total / 1e6, 2) == pr["flash_values_millions"]
    std = tiled.standard_attention_accesses(T, T, d)
    assert std == 4 * T * T + 4 * T * d == 4_456_448
    assert round(std / 1e6, 2) == pr["standard_values_millions"]
    assert res.tiles_total == pr["tiles_total"]
    rc_ = tiled.flash_forward(q, k, v, Br, Bc, causal=True)
    assert rc_.tiles_visited == pr["causal_tiles_visited"] == tiled.causal_tiles_visited(T, Br, Bc)
    # with n square blocks per side the visited fraction is n(n+1)/2 of n^2
    n = 16
    assert tiled.causal_tiles_visited(n * 64, 64, 64) == n * (n + 1) // 2


def test_io_theorem_shape():
    """FA1-order count ~ 12 T^2 d^2 / M for M >> d^2, and it loses to standard attention when
    M is near d^2 (zerotofrontier 12.3, 'The IO complexity theorem')."""
    T, d = 4096, 64
    M = 100_000
    Bc, Br = tiled.fa1_block_sizes(M, d)
    assert Bc == math.ceil(M / (4 * d)) and Br == min(Bc, d)
    fa1 = tiled.fa1_order_accesses(T, d, Bc)
    assert 0.8 < fa1 / (12 * T * T * d * d / M) < 1.25
    std = tiled.standard_attention_accesses(T, T, d)
    assert fa1 < std / 5
    Bc_small, _ = tiled.fa1_block_sizes(d * d, d)
    assert tiled.fa1_order_accesses(T, d, Bc_small) > std
    # FA2 order at B_r = 128: ~(2T/B_r + 2) T d values against 4T^2 + 4Td
    assert tiled.fa2_order_accesses(T, d, 128) < std / 3


def test_memory_arithmetic():
    g = json.load(open(os.path.join(GOLD, "memory_arithmetic.json")))
    L = g["llama_layer"]
    p_bytes, lse_bytes = tiled.saved_state_bytes(L["heads"], L["T"], p_bytes=2, lse_bytes=4)
    assert p_bytes == L["p_bytes_printed_gib"] * 2**30
    assert lse_bytes == L["lse_bytes_printed_mib"] * 2**20
    b = g["batch_scores"]
    assert b["B"] * b["H"] * b["T"] ** 2 * b["bytes_per_value"] == b["printed_gb"] * 2**30
    w = g["wide_tile"]
    assert w["rows"] * w["d"] * w["bytes_per_value"] == w["printed_bytes"]
