"""fp64 model of the tiled algorithm and its HBM-traffic counters -- TEST INFRASTRUCTURE ONLY.

This is the pages' own teaching model restated in numpy, used by the tests to
pin the online-softmax merge, the causal skip test and the IO counts that the
pages print.  It is not a reference for the CUDA path (that is the naive
oracle in ``attn_oracle.c``); it is itself compared against the naive oracle.

Sources:
  * zerotofrontier "FlashAttention" (Efficient attention 12.3): "The picture, a
    grid of tiles" (n_r = ceil(Tq/B_r), n_c = ceil(Tk/B_c)); "The forward pass"
    (steps 1-3, the unnormalised accumulator divided once at the end); "The
    causal mask, and the tiles you never visit" (three tile kinds, skip test
    first-key-of-block > last-query-of-block); "The backward pass, derived"
    (D preprocess, key blocks outside, dQ accumulated by read-add-write);
    "The IO complexity theorem" (FA2-order count Td + 2Td*n_r + Td + T, FA1
    order 2Td + n_c(3Td + 4T)).
  * "FlashAttention -- IO-Aware Exact Attention" (atlas wiki), "Standard
    attention, and why it's wasteful", and the hemanths blog "Standard
    Attention: What Actually Happens" (the S/P round trips of standard
    attention: 4T^2 + 4Td values).
  * llmdeepdive 7.7 "FlashAttention & IO-awareness", "01 Concept" (the worked
    example that the trace reproduces).

Causal alignment is bottom-right (key l allowed for row r iff l <= r + Tk - Tq),
the same reading as the oracle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass
class HBMCounter:
    """Counts values (not bytes) moved between HBM and on-chip memory."""
    reads: int = 0
    writes: int = 0

    def read(self, n: int) -> None:
        self.reads += int(n)

    def write(self, n: int) -> None:
        self.writes += int(n)

    @property
    def total(self) -> int:
        return self.reads + self.writes


@dataclass
class ForwardResult:
    o: np.ndarray
    lse: np.ndarray
    counter: HBMCounter
    tiles_visited: int
    tiles_total: int
    trace: list = field(default_factory=list)


def _mask(rows: np.ndarray, cols: np.ndarray, Tq: int, Tk: int) -> np.ndarray:
    """True where key cols[b] is allowed for query rows[a] (bottom-right causal)."""
    return cols[None, :] <= rows[:, None] + (Tk - Tq)


def flash_forward(Q, K, V, Br: int, Bc: int, causal: bool = False, scale: float | None = None,
                  trace_row: int | None = None) -> ForwardResult:
    """Query blocks outside, key/value blocks inside; O written once per block."""
    Q, K, V = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
    Tq, d = Q.shape
    Tk = K.shape[0]
    c = 1.0 / math.sqrt(d) if scale is None else float(scale)
    n_r, n_c = math.ceil(Tq / Br), math.ceil(Tk / Bc)
    O = np.zeros((Tq, V.shape[1]))
    lse = np.zeros(Tq)
    cnt = HBMCounter()
    visited = 0
    trace = []
    for i in range(n_r):
        rows = np.arange(i * Br, min((i + 1) * Br, Tq))
        Qi = Q[rows]
        cnt.read(Qi.size)                                   # step 1: load Q_i
        m = np.full(rows.size, -np.inf)
        ell = np.zeros(rows.size)
        Ot = np.zeros((rows.size, V.shape[1]))
        for j in range(n_c):
            j0 = j * Bc
            if causal and j0 > rows[-1] + (Tk - Tq):       # whole tile above the diagonal
                continue
            visited += 1
            cols = np.arange(j0, min(j0 + Bc, Tk))
            Kj, Vj = K[cols], V[cols]
            cnt.read(Kj.size + Vj.size)                     # step 2.1: load K_j, V_j
            S = c * (Qi @ Kj.T)                             # step 2.2
            if causal:
                S = np.where(_mask(rows, cols, Tq, Tk), S, -np.inf)
            m_new = np.maximum(m, S.max(axis=1))            # step 2.3
            ref = np.where(m_new == -np.inf, 0.0, m_new)    # rows with nothing allowed yet
            Pt = np.exp(S - ref[:, None])                   # step 2.4
            alpha = np.exp(m - ref)
            if trace_row is not None and trace_row in rows:
                a = int(np.where(rows == trace_row)[0][0])
                trace.append({"block": j, "m_old": m[a], "m_new": m_new[a],
                              "ell_rescaled": alpha[a] * ell[a],
                              "ell": alpha[a] * ell[a] + Pt[a].sum()})
            ell = alpha * ell + Pt.sum(axis=1)              # step 2.5
            Ot = alpha[:, None] * Ot + Pt @ Vj
            m = m_new
        live = ell > 0
        O[rows] = np.where(live[:, None], Ot / np.where(live, ell, 1.0)[:, None], 0.0)   # step 3
        lse[rows] = np.where(live, m + np.log(np.where(live, ell, 1.0)), -np.inf)
        cnt.write(O[rows].size + rows.size)                 # write O_i and lse_i once
    return ForwardResult(O, lse, cnt, visited, n_r * n_c, trace)


def flash_backward(Q, K, V, O, dO, lse, Br: int, Bc: int, causal: bool = False,
                   scale: float | None = None):
    """Key/value blocks outside; dK_j, dV_j accumulate on chip; dQ_i by read-add-write."""
    Q, K, V, O, dO, lse = (np.asarray(x, dtype=np.float64) for x in (Q, K, V, O, dO, lse))
    Tq, d = Q.shape
    Tk = K.shape[0]
    c = 1.0 / math.sqrt(d) if scale is None else float(scale)
    n_r, n_c = math.ceil(Tq / Br), math.ceil(Tk / Bc)
    cnt = HBMCounter()
    D = (dO * O).sum(axis=1)                                # preprocess: D_r = dO_r . O_r
    cnt.read(dO.size + O.size)
    cnt.write(D.size)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for j in range(n_c):
        j0 = j * Bc
        cols = np.arange(j0, min(j0 + Bc, Tk))
        Kj, Vj = K[cols], V[cols]
        cnt.read(Kj.size + Vj.size)
        dKj = np.zeros_like(Kj)
        dVj = np.zeros_like(Vj)
        for i in range(n_r):
            rows = np.arange(i * Br, min((i + 1) * Br, Tq))
            if causal and j0 > rows[-1] + (Tk - Tq):
                continue
            Qi, dOi = Q[rows], dO[rows]
            cnt.read(Qi.size + dOi.size + 2 * rows.size)    # Q_i, dO_i, lse_i, D_i
            S = c * (Qi @ Kj.T)
            lse_i = lse[rows]
            live = np.isfinite(lse_i)                       # rows with at least one key
            allowed = _mask(rows, cols, Tq, Tk) if causal else np.ones(S.shape, bool)
            allowed &= live[:, None]
            safe = np.where(live, lse_i, 0.0)[:, None]
            P = np.exp(np.where(allowed, S - safe, -np.inf))   # weights rebuilt from lse
            dVj += P.T @ dOi
            dP = dOi @ Vj.T
            dS = P * (dP - D[rows][:, None])
            cnt.read(rows.size * d)                         # dQ_i: read, add, write
            dQ[rows] += c * (dS @ Kj)
            cnt.write(rows.size * d)
            dKj += c * (dS.T @ Qi)
        dK[cols] = dKj
        dV[cols] = dVj
        cnt.write(dKj.size + dVj.size)
    return dQ, dK, dV, cnt


def standard_attention_accesses(Tq: int, Tk: int, d: int) -> int:
    """HBM values moved by standard attention: S and P round-trip through HBM.

    read Q, K; write S; read S; write P; read P, V; write O.
    """
    return (Tq * d + Tk * d) + Tq * Tk + Tq * Tk + Tq * Tk + (Tq * Tk + Tk * d) + Tq * d


def fa2_order_accesses(T: int, d: int, Br: int) -> int:
    """Query blocks outside: Td + 2Td*ceil(T/B_r) + Td + T."""
    return T * d + 2 * T * d * math.ceil(T / Br) + T * d + T


def fa1_order_accesses(T: int, d: int, Bc: int) -> int:
    """Key/value blocks outside: 2Td + n_c (3Td + 4T) with n_c = ceil(T/B_c)."""
    return 2 * T * d + math.ceil(T / Bc) * (3 * T * d + 4 * T)


def fa1_block_sizes(M: int, d: int) -> tuple[int, int]:
    """B_c = ceil(M / 4d), B_r = min(ceil(M / 4d), d)."""
    bc = math.ceil(M / (4 * d))
    return bc, min(bc, d)


def causal_tiles_visited(T: int, Br: int, Bc: int) -> int:
    """Tiles left after the skip test on a square causal grid."""
    n = 0
    for i in range(math.ceil(T / Br)):
        last = min((i + 1) * Br, T) - 1
        n += sum(1 for j in range(math.ceil(T / Bc)) if not j * Bc > last)
    return n


def saved_state_bytes(heads: int, T: int, p_bytes: int = 2, lse_bytes: int = 4) -> tuple[int, int]:
    """Bytes kept for the backward pass: the full P versus one lse per row."""
    return heads * T * T * p_bytes, heads * T * lse_bytes
