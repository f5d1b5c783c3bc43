#!/usr/bin/env python
"""Benchmark: attention fwd+bwd TFLOP/s, bf16, B8 H32 N4096 d128 causal, as a
fraction of the GB300 dense BF16 peak.

A step is one forward (fa_fwd) and one backward (fa_bwd: preprocess, tile
loop, dQ finish) over the whole workload, inputs resident in HBM.  FLOPs per
step: 4d (forward) + 10d (backward) per unmasked (query, key) pair, with a
causal square counted as T^2/2 pairs per head.  Inputs (q, k, v, dO: 4 x 268 MB
of bf16) are larger than the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torch.distributed.run, one rank per GPU, each rank running
the full workload on its own GPU (weak scaling, no data-path collective);
value is the sum over ranks divided by the slowest rank's time.  Rank 0
prints one JSON line.  --impl reference times the fp64 CPU oracle on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s fwd+bwd, bf16 B8 H32 N4096 d128 causal; % of BF16 peak"
WORKLOAD = dict(name="attention fwd+bwd B8 H32 N4096 d128 causal", B=8, H=32, T=4096, d=128, causal=True)
KERNELS_PER_STEP = 4   # fwd, bwd preprocess, bwd tile loop, bwd dQ finish


# ------------------------------------------------------------------ helpers
def flops_per_head(T: int, d: int, causal: bool) -> tuple[float, float]:
    pairs = T * T / 2 if causal else T * T
    return 4.0 * d * pairs, 10.0 * d * pairs


def step_flops(w=WORKLOAD) -> tuple[float, float]:
    f, b = flops_per_head(w["T"], w["d"], w["causal"])
    n = w["B"] * w["H"]
    return f * n, b * n


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"bf16_tflops": float(p["bf16_tflops"]), "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# Committed ncu summaries: (kernel, head width) -> (summary, the sources its hash covers).  A
# summary lists, per full-size workload it was scaled to, "dram-bytes-per-launch-<key>: N".
_FWD_SRC, _BWD_SRC = ("fa_fwd_sm103.cu", "fa_common.cuh"), ("fa_bwd_sm103.cu", "fa_common.cuh")
PROFILE_OF = {("bwd_main", 128): ("profiles/bwd_main_d128_b2h32_t4096_causal.md", _BWD_SRC),
              ("fwd", 128): ("profiles/fwd_kernel_d128_b2h32_t4096_causal.md", _FWD_SRC),
              ("fwd", 256): ("profiles/fwd_kernel_d256_b1h4_t32768_causal.md", _FWD_SRC),
              ("fwd", 64): ("profiles/fwd_kernel_d64_b1h6_t65536.md", _FWD_SRC),
              ("bwd_main", 64): ("profiles/bwd_main_d64_b1h6_t65536.md", _BWD_SRC)}


def ncu_traffic(kernel: str, d: int = 128, key: str = "b8h32") -> int | None:
    """DRAM bytes (read + write) per full-size launch of workload `key` from the committed ncu
    summary of `kernel` at head width d, or None: no such summary or figure, or the kernel's
    sources changed since that capture."""
    import hashlib
    import re
    if (kernel, d) not in PROFILE_OF:
        return None
    path, srcs = PROFILE_OF[(kernel, d)]
    try:
        text = open(os.path.join(ROOT, path)).read()
        h = hashlib.sha256()
        for f in srcs:
            h.update(open(os.path.join(ROOT, "exact_io_aware_05_gb300", "csrc", f), "rb").read())
        sha = re.search(r"source-sha256-16:\s*([0-9a-f]{16})", text)
        if sha.group(1) != h.hexdigest()[:16]:
            return None
        return int(re.search(rf"dram-bytes-per-launch-{re.escape(key)}:\s*(\d+)", text).group(1))
    except Exception:
        return None


def dist_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def reduce_max(value: float, world: int, device=None) -> float:
    """Max over ranks (a host-side reduction of timings, not a data-path collective)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "50"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle leg
def oracle_sample(min_seconds: float = 10.0, max_heads: int = 64) -> dict:
    """The fp64 oracle (as it stands) on whole heads of the workload: forward for every
    row, backward for every row and key.  Runs heads until min_seconds have passed."""
    import numpy as np
    import torch

    import oracle
    from exact_io_aware_05_gb300 import inputs

    w = WORKLOAD
    wl = inputs.small(1, 1, w["T"], w["T"], w["d"], w["causal"], seed=4, scale=1.0 / math.sqrt(w["d"]),
                      backward=True)
    cores = oracle.default_threads()
    f_head, b_head = flops_per_head(w["T"], w["d"], w["causal"])
    heads, t_total = 0, 0.0
    while heads < max_heads and (t_total < min_seconds or heads == 0):
        x = inputs.generate(inputs.replace(wl, seed=4 + heads))
        q, k, v, do = (x[n][0, 0].to(torch.float64).numpy() for n in ("q", "k", "v", "do"))
        t0 = time.perf_counter()
        oracle.attention_fwd(q, k, v, wl.causal, wl.scale, nthreads=cores)
        oracle.attention_bwd(q, k, v, do, wl.causal, wl.scale, nthreads=cores)
        t_total += time.perf_counter() - t0
        heads += 1
    tflops = heads * (f_head + b_head) / t_total / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{heads} of the {w['B'] * w['H']} heads (T={w['T']}, d={w['d']}, causal), forward every row "
                      f"+ backward every row and key, fp64, {t_total:.1f} s",
            "seconds": t_total}


def run_reference(args) -> None:
    rank, _, world = dist_info()
    if rank != 0:
        return
    import torch  # noqa: F401  (inputs module uses torch's CPU generator)

    import oracle
    from exact_io_aware_05_gb300 import inputs

    w = WORKLOAD
    wl = inputs.small(1, 1, w["T"], w["T"], w["d"], w["causal"], seed=4, scale=1.0 / math.sqrt(w["d"]),
                      backward=True)
    cores = oracle.default_threads()
    f_head, b_head = flops_per_head(w["T"], w["d"], w["causal"])
    x = inputs.generate(wl)
    import numpy as np  # noqa: F401
    q, k, v, do = (x[n][0, 0].to(torch.float64).numpy() for n in ("q", "k", "v", "do"))

    def one_step():
        oracle.attention_fwd(q, k, v, wl.causal, wl.scale, nthreads=cores)
        oracle.attention_bwd(q, k, v, do, wl.causal, wl.scale, nthreads=cores)

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = (time.perf_counter() - t0) / args.steps
    value = (f_head + b_head) / dt / 1e12
    sample = f"one head (T={w['T']}, d={w['d']}, causal) per step: forward every row + backward every row and key"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_block(world: int) -> dict:
    w = WORKLOAD
    return {"workload": w["name"], "B": w["B"], "H": w["H"], "N": w["T"], "d": w["d"], "causal": w["causal"],
            "flops": "4d fwd + 10d bwd per unmasked pair; causal square = T^2/2 pairs",
            "l2": "no flush: inputs q,k,v,dO = 4 x 268 MB bf16, larger than the 129 MB L2",
            "parallelism": f"replicas x{world} (one full workload per GPU, no data-path collective)"}


# ------------------------------------------------------------------ GPU leg
def run_ours(args) -> None:
    import torch

    rank, local, world = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from exact_io_aware_05_gb300 import fa

    w = WORKLOAD
    B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]
    scale = 1.0 / math.sqrt(d)
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + rank)
    shp = (B, H, T, d)
    q, k, v, do = (torch.randn(shp, device=dev, generator=g).to(torch.bfloat16) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, T), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = fa.alloc_workspace(B, H, T, T, d, dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        fa.fa_fwd(q, k, v, o, lse, causal, scale, stream)
        if evs is not None:
            evs[1].record(stream)
        fa.fa_bwd_stage(1, q, k, v, o, lse, do, dq, dk, dv, causal, scale, ws, stream)
        if evs is not None:
            evs[2].record(stream)
        fa.fa_bwd_stage(2, q, k, v, o, lse, do, dq, dk, dv, causal, scale, ws, stream)
        if evs is not None:
            evs[3].record(stream)
        fa.fa_bwd_stage(3, q, k, v, o, lse, do, dq, dk, dv, causal, scale, ws, stream)
        if evs is not None:
            evs[4].record(stream)

    for _ in range(args.warmup):
        step()
    if fa.fa_sync_status(stream) != fa.FA_OK:
        raise RuntimeError("device status error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
        time.sleep(0.3)   # let the sampler attach before the timed region
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    st = fa.fa_sync_status(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {st} after the timed region")

    total_ms = t_start.elapsed_time(t_end)
    ms_step = reduce_max(total_ms / args.steps, world, dev)
    per = [[e[i].elapsed_time(e[i + 1]) for i in range(4)] for e in evs]
    fwd_ms = statistics.mean(p[0] for p in per)
    pre_ms = statistics.mean(p[1] for p in per)
    main_ms = statistics.mean(p[2] for p in per)
    dq_ms = statistics.mean(p[3] for p in per)
    f_fwd, f_bwd = step_flops()
    value = world * (f_fwd + f_bwd) / (ms_step * 1e-3) / 1e12
    peaks = measured_peaks()
    peak = peaks["bf16_tflops"]
    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    main_tf = f_bwd / (main_ms * 1e-3) / 1e12
    bwd_tf = f_bwd / ((pre_ms + main_ms + dq_ms) * 1e-3) / 1e12
    dom = ("bwd_main", main_tf) if main_ms >= fwd_ms else ("fwd", fwd_tf)

    # e2e: the public API with host buffers, copies inside the timed region.  Every step
    # copies its own q, k, v, dO from pinned host memory and its o, lse, dq, dk, dv back;
    # with two device buffer sets the copies of neighbouring steps overlap the compute
    # (host-to-device on one stream, compute on the bench stream, device-to-host on a
    # third), as a training loop would stream batches.
    e2e = None
    if not args.no_e2e:
        pin = {n: t.to("cpu").pin_memory() for n, t in (("q", q), ("k", k), ("v", v), ("do", do))}
        outs = {n: torch.empty(shp, dtype=torch.bfloat16).pin_memory() for n in ("o", "dq", "dk", "dv")}
        out_lse = torch.empty((B, H, T), dtype=torch.float32).pin_memory()
        dbuf = [{n: torch.empty(shp, device=dev, dtype=torch.bfloat16) for n in ("q", "k", "v", "do")}
                for _ in range(2)]
        dout = [{n: torch.empty(shp, device=dev, dtype=torch.bfloat16) for n in ("o", "dq", "dk", "dv")}
                for _ in range(2)]
        dlse = [torch.empty((B, H, T), device=dev, dtype=torch.float32) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def run_e2e(n_steps, a0=None, a1=None):
            if a0 is not None:
                a0.record(s_in)
            for i in range(n_steps):
                b_ = i % 2
                x, y, yl = dbuf[b_], dout[b_], dlse[b_]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_comp[b_])      # compute i-2 is done with this input set
                    for n in ("q", "k", "v", "do"):
                        x[n].copy_(pin[n], non_blocking=True)
                    ev_in[b_].record(s_in)
                stream.wait_event(ev_in[b_])
                if i >= 2:
                    stream.wait_event(ev_out[b_])         # outputs of step i-2 have left the device
                fa.fa_fwd(x["q"], x["k"], x["v"], y["o"], yl, causal, scale, stream)
                fa.fa_bwd(x["q"], x["k"], x["v"], y["o"], yl, x["do"], y["dq"], y["dk"], y["dv"], causal, scale,
                          ws, stream)
                ev_comp[b_].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_comp[b_])
                    for n in ("o", "dq", "dk", "dv"):
                        outs[n].copy_(y[n], non_blocking=True)
                    out_lse.copy_(yl, non_blocking=True)
                    ev_out[b_].record(s_out)
            if a1 is not None:
                a1.record(s_out)

        run_e2e(2)
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(args.steps, 10))
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        run_e2e(n_e2e, a0, a1)
        torch.cuda.synchronize(dev)
        if fa.fa_sync_status(stream) != fa.FA_OK:
            raise RuntimeError("device status error in the end-to-end run")
        e2e_ms = reduce_max(a0.elapsed_time(a1) / n_e2e, world, dev)
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in outs.values()) + out_lse.numel() * 4
        e2e = {"value": world * (f_fwd + f_bwd) / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "api": "fa_fwd + fa_bwd with pinned host buffers, copies of neighbouring steps overlapped"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = oracle_sample(min_seconds=args.cpu_seconds)
        cpu = {k_: cb[k_] for k_ in ("value", "unit", "cores", "kind", "sample")}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(world),
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "passes": {"fwd": {"ms": fwd_ms, "tflops": fwd_tf, "pct_of_peak": 100 * fwd_tf / peak},
                   "bwd": {"ms": pre_ms + main_ms + dq_ms, "tflops": bwd_tf, "pct_of_peak": 100 * bwd_tf / peak,
                           "preprocess_ms": pre_ms, "tile_loop_ms": main_ms, "dq_finish_ms": dq_ms}},
        "roofline": {"kernel": dom[0], "bound": "tensor", "achieved": dom[1], "peak": peak, "unit": "TFLOP/s",
                     "frac": dom[1] / peak, "traffic": ncu_traffic(dom[0]) if WORKLOAD["B"] == 8 else None,
                     "peak_source": f"{peaks['source']} bf16 (burst), MEASURED_PEAKS.json"},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def run_decode(args) -> None:
    """Split-KV decode (fa_decode) on one GPU: one query row per sequence against a 32K-token
    key/value cache, B8 H32 d128.  HBM-bound: the metric is the K/V bytes streamed per second,
    against the measured HBM copy bandwidth.  A secondary line; the default run is the
    fwd+bwd workload above."""
    import torch
    from exact_io_aware_05_gb300 import fa, inputs
    w = inputs.WORKLOADS["decode_b8h32_q1_k32768_d128"]
    torch.cuda.set_device(0)
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    q = torch.randn(w.shape_q, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(w.shape_kv, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(w.shape_kv, device="cuda", generator=g).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(w.shape_q[:3], device="cuda")
    ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.H, w.Tq, w.Tk, w.d), dtype=torch.uint8, device="cuda")
    kv_bytes = 2 * k.numel() * k.element_size()
    step_bytes = kv_bytes + 2 * q.numel() * 2 + lse.numel() * 4
    for _ in range(args.warmup):
        fa.fa_decode(q, k, v, o, lse, w.causal, w.scale, ws)
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fa.fa_decode(q, k, v, o, lse, w.causal, w.scale, ws)
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    if fa.fa_sync_status() != fa.FA_OK:
        raise RuntimeError("fa_decode reported a device-side error")
    ms = e0.elapsed_time(e1) / args.steps
    gbs = step_bytes / (ms * 1e-3) / 1e9
    peak = measured_peaks().get("hbm_gbs")
    line = {"metric": "split-KV decode, K/V bytes streamed per second, bf16 B8 H32 Tq1 Tk32768 d128",
            "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Tq": w.Tq, "Tk": w.Tk, "d": w.d,
                       "causal": w.causal, "l2": "no flush: K and V are 4.3 GB, larger than the 129 MB L2"},
            "roofline": {"kernel": "decode_kernel + decode_merge_kernel", "bound": "hbm", "achieved": gbs,
                         "peak": peak, "unit": "GB/s", "frac": (gbs / peak) if peak else None,
                         "traffic": None, "peak_source": "measured HBM copy bandwidth, MEASURED_PEAKS.json"},
            "gpu_launches": 2 * args.steps, "clocks": clk}
    print(json.dumps(line), flush=True)


def run_fp8(args) -> None:
    """FP8 forward on one GPU, B8 H32 N4096 d128 causal: a step is fa_fp8_quantize (rotation,
    block scales, e4m3 codes from the bf16 q, k, v) then fa_fwd_fp8.  The metric is forward
    TFLOP/s (4d per unmasked pair) over the whole step; the forward kernel is also timed
    alone against the FP8 dense peak, taken as twice the measured bf16 peak (the nominal
    FP8 / BF16 ratio).  A secondary line; the default run is the bf16 fwd+bwd workload."""
    import torch
    from exact_io_aware_05_gb300 import fa, inputs
    w = inputs.WORKLOADS["fwd_fp8_b8h32_t4096_d128_causal"]
    if args.batch != w.B:   # a smaller batch, for profiling only
        w = inputs.replace(w, B=args.batch, name=f"fwd_fp8_b{args.batch}h32_t4096_d128_causal (profiling size)")
    torch.cuda.set_device(0)
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    q = torch.randn(w.shape_q, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(w.shape_kv, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(w.shape_kv, device="cuda", generator=g).to(torch.bfloat16)
    signs = inputs.rotation_signs(w.d, w.seed).cuda()
    o = torch.empty_like(q)
    lse = torch.empty(w.shape_q[:3], device="cuda")
    x = fa.alloc_fp8(w.B, w.H, w.Tq, w.Tk, w.d, "cuda")
    flops = 4.0 * w.d * w.Tq * w.Tq / 2 * w.B * w.H
    for _ in range(args.warmup):
        fa.fa_fp8_quantize(q, k, v, signs, out=x)
        fa.fa_fwd_fp8(x, o, lse, True, w.scale)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(0)
    clocks.start()
    for e in ev:
        e[0].record()
        fa.fa_fp8_quantize(q, k, v, signs, out=x)
        e[1].record()
        fa.fa_fwd_fp8(x, o, lse, True, w.scale)
        e[2].record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    if fa.fa_sync_status() != fa.FA_OK:
        raise RuntimeError("the FP8 forward reported a device-side error")
    ms = sum(e[0].elapsed_time(e[2]) for e in ev) / args.steps
    q_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    f_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    peaks = measured_peaks()
    peak8 = 2.0 * peaks["bf16_tflops"]
    fwd_tf = flops / (f_ms * 1e-3) / 1e12
    # quantization bytes: q, k, v read (v twice), codes written
    n = q.numel()
    qbytes = 2 * n * 3 + 2 * n + n * 3
    line = {"metric": "FP8 attention forward TFLOP/s (quantization included), B8 H32 N4096 d128 causal",
            "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.Tq, "d": w.d, "causal": True,
                       "rotation": "random signs + Hadamard", "l2": "no flush: q, k, v are 805 MB"},
            "split_ms": {"quantize": q_ms, "fwd_fp8": f_ms},
            "roofline": {"kernel": "fwd_kernel<128, false, true>", "bound": "tensor", "achieved": fwd_tf,
                         "peak": peak8, "unit": "TFLOP/s", "frac": fwd_tf / peak8, "traffic": None,
                         "peak_source": "2 x measured bf16 burst peak (nominal FP8/BF16 ratio), MEASURED_PEAKS.json"},
            "quantize_roofline": {"bound": "hbm", "achieved": qbytes / (q_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                                  "unit": "GB/s", "frac": qbytes / (q_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
            "gpu_launches": 5 * args.steps, "clocks": clk}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ per-workload lines
# The five configured workloads (inputs.WORKLOADS).  The default run above is the headline
# (B8 H32 N4096 d128 causal, forward + backward); --config N times workload N on its own and
# prints one contract line per variant.
CONFIG_SETS = {
    1: (["fwd_f32_b1h1_t256_d64"], "fwd"),
    2: (["fwd_b8h32_t4096_d128_causal", "fwd_b8h32_t4096_d128_causal_q4"], "fwd"),
    3: (["fwd_b1h24_t32768_d256_causal"], "fwd"),
    4: (["bwd_b8h32_t4096_d128_causal"], "bwd"),
    5: (["fwdbwd_b1h16_t65536_d64", "fwdbwd_b1h16_t65536_d64_causal", "fwdbwd_b1h16_q8192_k65536_d64_causal"],
        "fwdbwd"),
}
FP32_LANES_PER_SM = 128   # FP32 FMA lanes per SM (4 SMSPs x 32)


def _oracle_rows(w, rows, with_bwd: bool):
    """The fp64 oracle on the given rows of head 0 (forward; with_bwd: also the whole head's
    backward, every row and key): seconds and the flops of what it computed (4d per allowed
    pair of the rows forward, 10d per allowed pair of the head backward)."""
    import numpy as np
    import torch

    import oracle
    from exact_io_aware_05_gb300 import inputs

    x = inputs.generate(inputs.replace(w, B=1, H=1))
    q, k, v = (x[n][0, 0].to(torch.float64).numpy() for n in ("q", "k", "v"))
    cores = oracle.default_threads()
    off = w.Tk - w.Tq
    pairs = sum(min(w.Tk, max(0, int(r) + off + 1)) if w.causal else w.Tk for r in rows)
    t0 = time.perf_counter()
    oracle.attention_fwd(q, k, v, w.causal, w.scale, rows=np.asarray(rows), nthreads=cores)
    flops = 4.0 * w.d * pairs
    if with_bwd:
        do = x["do"][0, 0].to(torch.float64).numpy()
        oracle.attention_bwd(q, k, v, do, w.causal, w.scale, nthreads=cores)
        flops += 10.0 * w.d * inputs.allowed_pairs(w.Tq, w.Tk, w.causal)
    return time.perf_counter() - t0, flops, cores


def run_config(args) -> None:
    """Times one configured workload (each of its variants) on one GPU: the forward (fa_fwd, or
    fa_fwd_f32 for the fp32 workload) and/or the backward (fa_bwd's three stages), inputs in HBM,
    CUDA events over `steps` calls after `warmup`; the roofline is the pass that takes longest.
    An end-to-end figure goes through the same calls with pinned host buffers, copies inside
    the timed region; the oracle is timed on a bounded sample of rows."""
    import torch
    from exact_io_aware_05_gb300 import fa, inputs

    names, kind = CONFIG_SETS[args.config]
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peaks = measured_peaks()
    stream = torch.cuda.current_stream(dev)
    for name in names:
        w = inputs.WORKLOADS[name]
        if args.heads is not None:   # profiling size: fewer heads, same shape per head
            w = inputs.replace(w, H=args.heads, name=f"{w.name} (profiling size: H{args.heads})")
        f32 = w.dtype == torch.float32
        g = torch.Generator(device=dev)
        g.manual_seed(4321 + w.seed)
        shp_q, shp_k = w.shape_q, w.shape_kv
        q = torch.randn(shp_q, device=dev, generator=g) * w.q_scale
        k = torch.randn(shp_k, device=dev, generator=g)
        v = torch.randn(shp_k, device=dev, generator=g)
        do = torch.randn(shp_q, device=dev, generator=g)
        if not f32:
            q, k, v, do = (t.to(torch.bfloat16) for t in (q, k, v, do))
        o = torch.empty_like(q)
        lse = torch.empty(shp_q[:3], device=dev, dtype=torch.float32)
        BH = w.B * w.H
        pairs = inputs.allowed_pairs(w.Tq, w.Tk, w.causal) * BH
        f_fwd, f_bwd = 4.0 * w.d * pairs, 10.0 * w.d * pairs
        has_fwd, has_bwd = kind in ("fwd", "fwdbwd"), kind in ("bwd", "fwdbwd")
        ws = fa.alloc_workspace(w.B, w.H, w.Tq, w.Tk, w.d, dev) if has_bwd else None
        dq, dk, dv = (torch.empty_like(t) for t in (q, k, v)) if has_bwd else (None, None, None)
        # small inputs (the fp32 workload) sit in L2: a 256 MB buffer is written between calls
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if f32 else None

        def fwd():
            (fa.fa_fwd_f32 if f32 else fa.fa_fwd)(q, k, v, o, lse, w.causal, w.scale, stream)

        def bwd(st):
            fa.fa_bwd_stage(st, q, k, v, o, lse, do, dq, dk, dv, w.causal, w.scale, ws, stream)

        fwd()   # o, lse for the backward
        for _ in range(args.warmup):
            if has_fwd:
                fwd()
            if has_bwd:
                for st in (1, 2, 3):
                    bwd(st)
        torch.cuda.synchronize(dev)
        if fa.fa_sync_status(stream) != fa.FA_OK:
            raise RuntimeError(f"{name}: device status error during warm-up")
        sampler = ClockSampler(0)
        sampler.start()
        time.sleep(0.3)
        t_f, t_pre, t_main, t_dq = [], [], [], []
        for _ in range(args.steps):
            if flush is not None:
                flush.fill_(1)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            ev[0].record(stream)
            if has_fwd:
                fwd()
            ev[1].record(stream)
            if has_bwd:
                bwd(1)
                ev[2].record(stream)
                bwd(2)
                ev[3].record(stream)
                bwd(3)
            ev[4].record(stream)
            torch.cuda.synchronize(dev)
            t_f.append(ev[0].elapsed_time(ev[1]))
            if has_bwd:
                t_pre.append(ev[1].elapsed_time(ev[2]))
                t_main.append(ev[2].elapsed_time(ev[3]))
                t_dq.append(ev[3].elapsed_time(ev[4]))
        clocks = sampler.stop()
        if fa.fa_sync_status(stream) != fa.FA_OK:
            raise RuntimeError(f"{name}: device status error in the timed region")
        med = statistics.median
        fwd_ms = med(t_f) if has_fwd else 0.0
        bwd_ms = (med(t_pre) + med(t_main) + med(t_dq)) if has_bwd else 0.0
        flops = (f_fwd if has_fwd else 0.0) + (f_bwd if has_bwd else 0.0)
        ms = fwd_ms + bwd_ms
        value = flops / (ms * 1e-3) / 1e12
        passes = {}
        if has_fwd:
            passes["fwd"] = {"ms": fwd_ms, "tflops": f_fwd / (fwd_ms * 1e-3) / 1e12}
        if has_bwd:
            passes["bwd"] = {"ms": bwd_ms, "tflops": f_bwd / (bwd_ms * 1e-3) / 1e12, "preprocess_ms": med(t_pre),
                             "tile_loop_ms": med(t_main), "dq_finish_ms": med(t_dq)}
        if f32:
            peak = 2.0 * FP32_LANES_PER_SM * torch.cuda.get_device_properties(dev).multi_processor_count * \
                (clocks["sm_max_mhz"] if clocks and clocks.get("sm_max_mhz") else 2070.0) * 1e6 / 1e12
            roof = {"kernel": "fwd_f32_kernel", "bound": "alu", "achieved": passes["fwd"]["tflops"], "peak": peak,
                    "unit": "TFLOP/s", "frac": passes["fwd"]["tflops"] / peak, "traffic": None,
                    "peak_source": "derived: SMs x 128 FP32 lanes x 2 flops x max SM clock (fp32 FFMA)"}
        else:
            peak = peaks["bf16_tflops"]
            if has_bwd and (not has_fwd or med(t_main) >= fwd_ms):
                dom = ("bwd_main", f_bwd / (med(t_main) * 1e-3) / 1e12)
            else:
                dom = ("fwd", passes["fwd"]["tflops"])
            roof = {"kernel": dom[0], "bound": "tensor", "achieved": dom[1], "peak": peak, "unit": "TFLOP/s",
                    "frac": dom[1] / peak, "traffic": ncu_traffic(dom[0], w.d, w.name) if args.heads is None else None,
                    "peak_source": f"{peaks['source']} bf16 (burst), MEASURED_PEAKS.json"}
        # end to end: the same calls with the inputs copied in from pinned host memory and the
        # outputs copied back, all inside the timed region
        e2e = None
        if not args.no_e2e:
            # inputs: q, k, v (+ dO; the backward-only workload also takes the forward's o, lse)
            ins = [("q", q), ("k", k), ("v", v)] + ([("do", do)] if has_bwd else []) + \
                  ([("o", o), ("lse", lse)] if not has_fwd else [])
            hin = {n: t.to("cpu").pin_memory() for n, t in ins}
            outs = ([("o", o), ("lse", lse)] if has_fwd else []) + ([("dq", dq), ("dk", dk), ("dv", dv)] if has_bwd else [])
            hout = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in outs}
            dev_in = dict(ins)
            dev_out = dict(outs)
            n_e2e = max(3, min(args.steps, 10))
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(n_e2e):
                for n, t in hin.items():
                    dev_in[n].copy_(t, non_blocking=True)
                if has_fwd:
                    fwd()
                if has_bwd:
                    fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, w.causal, w.scale, ws, stream)
                for n, t in hout.items():
                    t.copy_(dev_out[n], non_blocking=True)
            a1.record(stream)
            torch.cuda.synchronize(dev)
            e2e_ms = a0.elapsed_time(a1) / n_e2e
            e2e = {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                   "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin.values()),
                   "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout.values()),
                   "ms_per_step": e2e_ms,
                   "api": {"fwd": "fa_fwd", "bwd": "fa_bwd (o, lse copied in with the inputs)",
                           "fwdbwd": "fa_fwd + fa_bwd"}[kind] + " with pinned host buffers"}
        cpu = None
        if not args.no_cpu_baseline:
            import numpy as np
            nrow = w.Tq if w.Tq * w.Tk <= 1 << 24 else 1024
            rows = np.arange(w.Tq) if nrow == w.Tq else np.linspace(0, w.Tq - 1, nrow).astype(np.int64)
            secs, fl, cores = _oracle_rows(w, rows, has_bwd and w.Tk <= 8192)
            part = "forward every row" if nrow == w.Tq else f"forward of {nrow} rows spread over head 0"
            if has_bwd and w.Tk <= 8192:
                part += " + backward of the whole head (every row and key)"
            cpu = {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                   "sample": f"{part}, fp64, {secs:.2f} s; rate over the flops it computed" +
                             ("" if nrow == w.Tq else " (extrapolates to the whole workload by pair count)")}
        metric = {"fwd": "attention forward TFLOP/s", "bwd": "attention backward TFLOP/s",
                  "fwdbwd": "attention TFLOP/s fwd+bwd"}[kind]
        line = {"metric": f"{metric}, {'fp32' if f32 else 'bf16'} B{w.B} H{w.H} Tq{w.Tq} Tk{w.Tk} d{w.d} "
                          f"{'causal' if w.causal else 'non-causal'}" + (f", Q x{w.q_scale:g}" if w.q_scale != 1 else ""),
                "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32" if f32 else "bf16", "data": "synthetic",
                "config": {"workload": w.name, "B": w.B, "H": w.H, "Tq": w.Tq, "Tk": w.Tk, "d": w.d,
                           "causal": w.causal, "q_scale": w.q_scale,
                           "flops": "4d fwd + 10d bwd per allowed pair (bottom-right causal)",
                           "l2": "256 MB written between calls" if f32 else "no flush: inputs larger than the 129 MB L2"},
                "pct_of_peak": 100.0 * value / peak, "passes": passes, "roofline": roof,
                "gpu_launches": (1 if has_fwd else 0) * args.steps + (3 if has_bwd else 0) * args.steps,
                "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks}
        print(json.dumps(line), flush=True)
        del q, k, v, do, o, lse, ws, dq, dk, dv, flush
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode", action="store_true",
                    help="time split-KV decode (B8 H32 Tq1 Tk32768 d128) instead of the fwd+bwd step")
    ap.add_argument("--fp8", action="store_true",
                    help="time the FP8 forward (quantization + fa_fwd_fp8, B8 H32 N4096 d128 causal)")
    ap.add_argument("--config", type=int, choices=sorted(CONFIG_SETS), default=None,
                    help="time configured workload 1..5 (each variant) instead of the headline step")
    ap.add_argument("--batch", type=int, default=WORKLOAD["B"],
                    help="batch size (default 8, the benchmark workload; smaller only for profiling)")
    ap.add_argument("--heads", type=int, default=None,
                    help="with --config: heads per workload (default: the workload's; fewer only for profiling)")
    args = ap.parse_args()
    if args.batch != WORKLOAD["B"]:
        WORKLOAD["B"] = args.batch
        WORKLOAD["name"] = f"attention fwd+bwd B{args.batch} H32 N4096 d128 causal (profiling size)"
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.config is not None:
        run_config(args)
    elif args.decode:
        run_decode(args)
    elif args.fp8:
        run_fp8(args)
    else:
        run_ours(args)
    if dist_info()[2] > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
