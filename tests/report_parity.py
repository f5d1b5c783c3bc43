"""Parity report of the five configured workloads (not a test: run it as a script on a GPU).

For each workload, the CUDA path through the C ABI and the fp64 oracle on the same seeded
inputs and the same samples as the parity tests (test_fwd_gpu.py, test_bwd_gpu.py): 8 heads
of the 4096/d128 forward, 4 heads of its backward, 512 rows x 4 heads at 32K/d256, 256 rows
(forward) and 48 rows / 48 keys (backward) of one head at 64K/d64.  Prints one JSON line per
workload with, for each output, the raw max |gpu - oracle| and the error beyond half a bf16
ulp of the exact value (the output format's own rounding), and for O also the raw maximum
over the elements with |O| < 2, where half an ulp is at most 2^-9 so that a bf16 output can
meet 1e-2 outright.

    python tests/report_parity.py [--workloads name,name,...]
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from exact_io_aware_05_gb300 import inputs  # noqa: E402
from gpu_util import excess_over_output_rounding, heads_of, rows_of, to64  # noqa: E402

FWD = {"fwd_f32_b1h1_t256_d64": (1, None), "fwd_b8h32_t4096_d128_causal": (8, None),
       "fwd_b8h32_t4096_d128_causal_q4": (8, None), "fwd_b1h24_t32768_d256_causal": (4, 512),
       "fwdbwd_b1h16_t65536_d64": (2, 256), "fwdbwd_b1h16_t65536_d64_causal": (2, 256),
       "fwdbwd_b1h16_q8192_k65536_d64_causal": (2, 256)}
BWD = {"bwd_b8h32_t4096_d128_causal": (4, None, None), "fwdbwd_b1h16_t65536_d64": (1, 48, 48),
       "fwdbwd_b1h16_t65536_d64_causal": (1, 48, 48), "fwdbwd_b1h16_q8192_k65536_d64_causal": (1, 48, 48)}


def forward_report(fa, w, nheads, nrows):
    x = inputs.generate(w, with_grad=False, device="cuda")
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.causal, w.scale)
    assert fa.fa_sync_status() == fa.FA_OK
    rows = None if nrows is None else rows_of(w.Tq, nrows)
    r = {"o_raw": 0.0, "o_beyond_rounding": -np.inf, "o_raw_where_abs_lt_2": 0.0, "lse_raw": 0.0}
    t0 = time.perf_counter()
    for (b, h) in heads_of(w, nheads):
        q, k, v = (to64(x[n][b, h]) for n in ("q", "k", "v"))
        o_ref, lse_ref = oracle.attention_fwd(q, k, v, w.causal, w.scale, rows=rows)
        og = to64(o[b, h]) if rows is None else to64(o[b, h])[rows]
        lg = to64(lse[b, h]) if rows is None else to64(lse[b, h])[rows]
        live = np.isfinite(lse_ref)
        err = np.abs(og - o_ref)
        r["o_raw"] = max(r["o_raw"], float(err.max()))
        r["o_beyond_rounding"] = max(r["o_beyond_rounding"], excess_over_output_rounding(og, o_ref))
        small = np.abs(o_ref) < 2
        if small.any():
            r["o_raw_where_abs_lt_2"] = max(r["o_raw_where_abs_lt_2"], float(err[small].max()))
        if live.any():
            r["lse_raw"] = max(r["lse_raw"], float(np.abs(lg[live] - lse_ref[live]).max()))
    r["oracle_seconds"] = time.perf_counter() - t0
    r["sample"] = f"{nheads} heads" + ("" if rows is None else f" x {len(rows)} rows")
    return r


def backward_report(fa, w, nheads, nrows, nkeys):
    x = inputs.generate(w, with_grad=True, device="cuda")
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.causal, w.scale)
    dq, dk, dv = fa.attention_backward(x["q"], x["k"], x["v"], o, lse, x["do"], w.causal, w.scale)
    assert fa.fa_sync_status() == fa.FA_OK
    rows = None if nrows is None else rows_of(w.Tq, nrows)
    keys = None if nkeys is None else rows_of(w.Tk, nkeys, seed=1)
    r = {f"{n}_{k_}": 0.0 for n in ("dq", "dk", "dv") for k_ in ("raw", "beyond_rounding")}
    t0 = time.perf_counter()
    for (b, h) in heads_of(w, nheads):
        q, k, v, do = (to64(x[n][b, h]) for n in ("q", "k", "v", "do"))
        ref = oracle.attention_bwd(q, k, v, do, w.causal, w.scale, rows=rows, keys=keys)
        for n, t, ix in (("dq", dq, rows), ("dk", dk, keys), ("dv", dv, keys)):
            g = to64(t[b, h]) if ix is None else to64(t[b, h])[ix]
            r[f"{n}_raw"] = max(r[f"{n}_raw"], float(np.abs(g - ref[n]).max()))
            r[f"{n}_beyond_rounding"] = max(r[f"{n}_beyond_rounding"], excess_over_output_rounding(g, ref[n]))
    r["oracle_seconds"] = time.perf_counter() - t0
    r["sample"] = f"{nheads} heads" + ("" if rows is None else f", {len(rows)} rows, {len(keys)} keys")
    return r


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", default=",".join(dict.fromkeys(list(FWD) + list(BWD))))
    args = ap.parse_args()
    from exact_io_aware_05_gb300 import fa
    for name in args.workloads.split(","):
        w = inputs.WORKLOADS[name]
        line = {"workload": name, "cores": oracle.default_threads()}
        if name in FWD:
            line["forward"] = forward_report(fa, w, *FWD[name])
        if name in BWD:
            line["backward"] = backward_report(fa, w, *BWD[name])
        print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
