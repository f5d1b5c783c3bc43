"""Seeded synthetic inputs and the workload table.

This module draws random numbers and describes shapes; it holds none of the
attention arithmetic, imports nothing from the CUDA binding or the oracle,
and is the one module both sides use.  Every tensor is drawn on the CPU with
a ``torch.Generator`` seeded per workload, as i.i.d. N(0, 1) fp32 values,
multiplied by ``q_scale`` (queries only) and then cast to the workload's
dtype.  The oracle reads back the same rounded values, so both sides see
bit-identical inputs.

The five workloads follow the attention shapes the pages discuss (batch,
heads, sequence length, head width) and the benchmark table of this library:
a tiny fp32 forward, the B8 H32 N4096 d128 causal forward and backward, a
wide-head (d=256) 32K forward, and a 64K long-context forward+backward with a
rectangular bottom-right causal case.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Tq: int
    Tk: int
    d: int
    causal: bool
    scale: float
    dtype: torch.dtype
    seed: int
    q_scale: float = 1.0
    backward: bool = False

    @property
    def shape_q(self):
        return (self.B, self.H, self.Tq, self.d)

    @property
    def shape_kv(self):
        return (self.B, self.H, self.Tk, self.d)

    def pairs(self) -> int:
        """Unmasked (query, key) pairs per head, bottom-right causal alignment."""
        return allowed_pairs(self.Tq, self.Tk, self.causal)


def allowed_pairs(Tq: int, Tk: int, causal: bool) -> int:
    """Unmasked (query, key) pairs of one head; row r sees keys l <= r + Tk - Tq when causal."""
    if not causal:
        return Tq * Tk
    off = Tk - Tq
    return sum(min(Tk, max(0, r + off + 1)) for r in range(Tq))


WORKLOADS = {
    "fwd_f32_b1h1_t256_d64": Workload("fwd_f32_b1h1_t256_d64", 1, 1, 256, 256, 64, False,
                                      1.0 / 8.0, torch.float32, seed=0),
    "fwd_b8h32_t4096_d128_causal": Workload("fwd_b8h32_t4096_d128_causal", 8, 32, 4096, 4096, 128,
                                            True, 1.0 / math.sqrt(128), torch.bfloat16, seed=1),
    "fwd_b8h32_t4096_d128_causal_q4": Workload("fwd_b8h32_t4096_d128_causal_q4", 8, 32, 4096, 4096,
                                               128, True, 1.0 / math.sqrt(128), torch.bfloat16,
                                               seed=2, q_scale=4.0),
    "fwd_b1h24_t32768_d256_causal": Workload("fwd_b1h24_t32768_d256_causal", 1, 24, 32768, 32768,
                                             256, True, 1.0 / 16.0, torch.bfloat16, seed=3),
    "bwd_b8h32_t4096_d128_causal": Workload("bwd_b8h32_t4096_d128_causal", 8, 32, 4096, 4096, 128,
                                            True, 1.0 / math.sqrt(128), torch.bfloat16, seed=4,
                                            backward=True),
    "fwdbwd_b1h16_t65536_d64": Workload("fwdbwd_b1h16_t65536_d64", 1, 16, 65536, 65536, 64, False,
                                        1.0 / 8.0, torch.bfloat16, seed=5, backward=True),
    "fwdbwd_b1h16_t65536_d64_causal": Workload("fwdbwd_b1h16_t65536_d64_causal", 1, 16, 65536,
                                               65536, 64, True, 1.0 / 8.0, torch.bfloat16, seed=5,
                                               backward=True),
    "fwdbwd_b1h16_q8192_k65536_d64_causal": Workload("fwdbwd_b1h16_q8192_k65536_d64_causal", 1, 16,
                                                     8192, 65536, 64, True, 1.0 / 8.0,
                                                     torch.bfloat16, seed=5, backward=True),
    # split-KV decode: one new query row per sequence against a 32K-token key/value cache
    # (bottom-right causal: the new row sees the whole cache), and 4 rows at 128K keys
    "decode_b8h32_q1_k32768_d128": Workload("decode_b8h32_q1_k32768_d128", 8, 32, 1, 32768, 128, True,
                                            1.0 / 128 ** 0.5, torch.bfloat16, seed=6),
    # FP8 forward (quantized inside the path) on the 4096/d128 shape, the same inputs as the
    # bf16 forward of that shape
    "fwd_fp8_b8h32_t4096_d128_causal": Workload("fwd_fp8_b8h32_t4096_d128_causal", 8, 32, 4096, 4096, 128,
                                                True, 1.0 / math.sqrt(128), torch.bfloat16, seed=1),
    "decode_b1h32_q4_k131072_d128": Workload("decode_b1h32_q4_k131072_d128", 1, 32, 4, 131072, 128, True,
                                             1.0 / 128 ** 0.5, torch.bfloat16, seed=7),
}


def small(B, H, Tq, Tk, d, causal, seed, dtype=torch.bfloat16, scale=None, q_scale=1.0,
          backward=False) -> Workload:
    """An ad-hoc workload for edge and ragged-shape tests."""
    return Workload(f"adhoc_b{B}h{H}_q{Tq}_k{Tk}_d{d}_{'c' if causal else 'n'}", B, H, Tq, Tk, d,
                    causal, (1.0 / math.sqrt(d)) if scale is None else scale, dtype, seed,
                    q_scale, backward)


def generate(w: Workload, with_grad: bool | None = None, device: str = "cpu"):
    """q, k, v (and dO if the workload has a backward pass), drawn in that order."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = torch.randn(w.shape_q, generator=g, dtype=torch.float32)
    if w.q_scale != 1.0:
        q.mul_(w.q_scale)
    k = torch.randn(w.shape_kv, generator=g, dtype=torch.float32)
    v = torch.randn(w.shape_kv, generator=g, dtype=torch.float32)
    out = {"q": q.to(w.dtype), "k": k.to(w.dtype), "v": v.to(w.dtype)}
    if w.backward if with_grad is None else with_grad:
        out["do"] = torch.randn(w.shape_q, generator=g, dtype=torch.float32).to(w.dtype)
    if device != "cpu":
        out = {n: t.to(device) for n, t in out.items()}
    return out


def rotation_signs(d: int, seed: int) -> torch.Tensor:
    """The FP8 forward's random rotation signs: d values +1.0 / -1.0 (fp32), each drawn
    as a fair bit by a torch.Generator seeded with `seed`."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randint(0, 2, (d,), generator=g).to(torch.float32) * 2.0 - 1.0


__all__ = ["Workload", "WORKLOADS", "allowed_pairs", "generate", "rotation_signs", "small", "replace"]
