"""Seeded synthetic inputs and the named workloads, shared by tests and bench.

This module holds no attention arithmetic: it only draws the random tensors
and names the shapes. Both the CUDA path and the CPU oracle are fed the same
rounded bits from here.

Recipe: a CPU ``torch.Generator`` seeded with the workload's seed draws, in
this order, Q, K, V and dO as float32 N(0, 1) (Q and K multiplied by the
workload's ``qk_mult`` before rounding), and each is rounded to the
workload's dtype (round-to-nearest-even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Tq: int
    Tkv: int
    D: int
    dtype: str          # "fp16" | "bf16"
    causal: bool
    window: int = 0
    qk_mult: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    # GQA 2:1 smoke shape, causal, fp16.
    "c1_b1_h2x1_t64_d64_fp16_causal": Workload(
        "c1_b1_h2x1_t64_d64_fp16_causal", 1, 2, 1, 64, 64, 64, "fp16", True, seed=0),
    # MHA, non-causal, bf16.
    "c2_b2_h8x8_t1024_d128_bf16": Workload(
        "c2_b2_h8x8_t1024_d128_bf16", 2, 8, 8, 1024, 1024, 128, "bf16", False, seed=1),
    # GQA 4:1, causal, the headline throughput workload.
    "c3_b4_h32x8_t4096_d128_bf16_causal": Workload(
        "c3_b4_h32x8_t4096_d128_bf16_causal", 4, 32, 8, 4096, 4096, 128, "bf16", True, seed=2),
    # GQA 8:1, causal + sliding window 4096, sharper softmax (Q, K x2).
    "c4_b1_h16x2_t16384_d128_bf16_causal_w4096": Workload(
        "c4_b1_h16x2_t16384_d128_bf16_causal_w4096", 1, 16, 2, 16384, 16384, 128, "bf16",
        True, window=4096, qk_mult=2.0, seed=3),
    # Shape sweep (fp16).
    "c5a_b2_h8x2_t2048_d64_fp16_causal": Workload(
        "c5a_b2_h8x2_t2048_d64_fp16_causal", 2, 8, 2, 2048, 2048, 64, "fp16", True, seed=5),
    "c5b_b2_h8x2_t2048_d96_fp16_causal": Workload(
        "c5b_b2_h8x2_t2048_d96_fp16_causal", 2, 8, 2, 2048, 2048, 96, "fp16", True, seed=6),
    "c5c_b2_h8x2_t2048_d256_fp16_causal": Workload(
        "c5c_b2_h8x2_t2048_d256_fp16_causal", 2, 8, 2, 2048, 2048, 256, "fp16", True, seed=7),
    "c5d_b2_h8x2_tq512_tkv2048_d128_fp16": Workload(
        "c5d_b2_h8x2_tq512_tkv2048_d128_fp16", 2, 8, 2, 512, 2048, 128, "fp16", False, seed=8),
    "c5e1_b2_h8x2_tq1_tkv1024_d128_fp16": Workload(
        "c5e1_b2_h8x2_tq1_tkv1024_d128_fp16", 2, 8, 2, 1, 1024, 128, "fp16", False, seed=9),
    "c5e4_b2_h8x2_tq4_tkv1024_d128_fp16": Workload(
        "c5e4_b2_h8x2_tq4_tkv1024_d128_fp16", 2, 8, 2, 4, 1024, 128, "fp16", False, seed=10),
    "c5e8_b2_h8x2_tq8_tkv1024_d128_fp16": Workload(
        "c5e8_b2_h8x2_tq8_tkv1024_d128_fp16", 2, 8, 2, 8, 1024, 128, "fp16", False, seed=11),
}

HEADLINE = "c3_b4_h32x8_t4096_d128_bf16_causal"


def make_inputs(w: Workload, with_do: bool = True) -> dict[str, torch.Tensor]:
    """Draw Q, K, V (and dO) on the CPU for workload ``w``, rounded to its dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    dt = w.torch_dtype
    q = torch.randn((w.B, w.Hq, w.Tq, w.D), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Hkv, w.Tkv, w.D), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Hkv, w.Tkv, w.D), generator=g, dtype=torch.float32)
    if w.qk_mult != 1.0:
        q.mul_(w.qk_mult)
        k.mul_(w.qk_mult)
    out = {"q": q.to(dt), "k": k.to(dt), "v": v.to(dt)}
    if with_do:
        out["do"] = torch.randn((w.B, w.Hq, w.Tq, w.D), generator=g,
                                dtype=torch.float32).to(dt)
    return out


def group_slice(t: torch.Tensor, b: int, h0: int, h1: int) -> torch.Tensor:
    """[B,H,T,D] -> [1, h1-h0, T, D] slice (a contiguous copy)."""
    return t[b:b + 1, h0:h1].contiguous()
