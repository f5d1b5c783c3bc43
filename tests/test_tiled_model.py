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


def test_fa1_order_count_by_hand():
    """The FA1-order count (key blocks outside) against loads and stores enumerated by hand
    on a 4 x 4 grid of tiles: zerotofrontier "FlashAttention", "The IO complexity theorem"
    (each K_j, V_j loaded once; per key block, each query block loads Q_i, O_i, l_i, m_i and
    writes O_i, l_i, m_i back).  T = 8, d = 2, B_c = 2 (n_c = 4), query blocks of 2 rows:
      K_j, V_j loads: 4 key blocks x (2 x 2 + 2 x 2)                 =  32
      per (i, j): loads Q_i 4 + O_i 4 + l_i 2 + m_i 2 = 12,
                  stores O_i 4 + l_i 2 + m_i 2 = 8;   16 tiles x 20  = 320
    total 352.  Ragged: T = 5, d = 3, B_c = 2 (n_c = 3): K, V 2 x 5 x 3 = 30; each sweep
    loads Q 15 + O 15 + l 5 + m 5 and stores O 15 + l 5 + m 5 = 65; 3 sweeps = 195; total 225."""
    assert tiled.fa1_order_accesses(8, 2, 2) == 32 + 16 * (12 + 8) == 352
    assert tiled.fa1_order_accesses(5, 3, 2) == 30 + 3 * 65 == 225
    # one block holds every key: a single sweep, K and V loaded once
    assert tiled.fa1_order_accesses(8, 2, 8) == 32 + (3 * 16 + 4 * 8) == 112


# Backward traffic enumerated by hand (zerotofrontier "FlashAttention", "The backward pass,
# derived": D in one pass over dO and O; key blocks outside, each K_j, V_j loaded once, dK_j,
# dV_j written once; per visited tile Q_i, dO_i, lse_i, D_i loaded and dQ_i read, added to
# and written back).  Each case: (Tq, Tk, d, Br, Bc, causal, reads, writes, tiles visited).
BWD_HAND = [
    # T = 8, d = 2, 4 x 4 blocks, 2 x 2 tiles.  reads: dO 16 + O 16; per key block K 8 + V 8;
    # per tile Q 8 + dO 8 + lse 4 + D 4 + dQ 8 = 32.  writes: D 8; per tile dQ 8; per key
    # block dK 8 + dV 8.  Non-causal, 4 tiles: reads 32 + 2 x 16 + 4 x 32 = 192,
    # writes 8 + 4 x 8 + 2 x 16 = 72.
    (8, 8, 2, 4, 4, False, 192, 72, 4),
    # causal: tile (query block 0, key block 1) is skipped (first key 4 > last row 3), 3 tiles:
    # reads 32 + 32 + 3 x 32 = 160, writes 8 + 3 x 8 + 32 = 64
    (8, 8, 2, 4, 4, True, 160, 64, 3),
    # Tq = 6, Tk = 10, bottom-right causal (offset 4), d = 2, 4 x 4 blocks with ragged tails.
    # Query block 0 (rows 0-3, last allowed key 7) skips key block 2 (keys 8-9); query block 1
    # (rows 4-5) sees all three.  reads: dO 12 + O 12; K, V 16 + 16 + 8; tiles of 4 rows
    # 4 x (2 + 2 + 1 + 1 + 2) = 32 (two of them), of 2 rows 16 (three): 24 + 40 + 64 + 48 = 176.
    # writes: D 6; dQ 8 + 8 + 4 + 4 + 4 = 28; dK, dV 16 + 16 + 8 = 40: 74.
    (6, 10, 2, 4, 4, True, 176, 74, 5),
]


@pytest.mark.parametrize("Tq,Tk,d,Br,Bc,causal,reads,writes,tiles", BWD_HAND)
def test_backward_counter_by_hand(Tq, Tk, d, Br, Bc, causal, reads, writes, tiles):
    q, k, v, dO = _inputs(Tq, Tk, d, seed=3, dO=True)
    g = oracle.attention_bwd(q, k, v, dO, causal, 0.5, want_o=True)
    *_, cnt = tiled.flash_backward(q, k, v, g["o"], dO, g["lse"], Br, Bc, causal, 0.5)
    assert (cnt.reads, cnt.writes) == (reads, writes)
    assert tiles == sum(1 for i in range(math.ceil(Tq / Br)) for j in range(math.ceil(Tk / Bc))
                        if not (causal and j * Bc > min((i + 1) * Br, Tq) - 1 + Tk - Tq))


def test_backward_traffic_has_no_square_term():
    """zerotofrontier "The backward pass, derived": the backward's traffic is a few dozen
    times T d, with no T^2 term.  At fixed block sizes the count per T d grows with the
    number of key blocks only (T / B_c), never with T^2 / d."""
    d, Br, Bc = 64, 128, 64
    per_td = []
    for T in (512, 1024):
        q, k, v, dO = _inputs(T, T, d, seed=T, dO=True)
        g = oracle.attention_bwd(q, k, v, dO, False, 0.125, want_o=True)
        *_, cnt = tiled.flash_backward(q, k, v, g["o"], dO, g["lse"], Br, Bc, False, 0.125)
        per_td.append(cnt.total / (T * d))
        # exact: D pass 2Td + T; K, V 2Td; n_c sweeps of (4Td + 2T); dK, dV 2Td
        n_c = T // Bc
        assert cnt.total == 2 * T * d + T + 2 * T * d + n_c * (4 * T * d + 2 * T) + 2 * T * d
    assert 12 < per_td[0] < per_td[1] < 100   # "a few dozen times T d"
