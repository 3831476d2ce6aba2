"""Seeded synthetic workloads for causal prefill attention.

This module only draws inputs. It holds none of the attention or quantisation
arithmetic, so both the CPU oracle and the CUDA path can take their inputs
from it without sharing any of the method's code.

The shapes follow the workloads of the ZYFA post ("Fast and Accurate FP8
Attention on AMD MI355X", sections "Throughput on Gaussian Inputs" and
"Throughput on Captured Activations at Sustained Clocks"): Gaussian Q/K/V at
head dimension 128 with grouped-query heads, the MLA head shape
(query-key dim 192, value dim 128), and activation-like inputs that stand in
for the captured Mistral-7B / Qwen3-8B layers (weights and text corpora are
not available, so outlier channels and RoPE imitate post-RoPE activations).

Recipe (identical on every machine, CPU generator, seed 0 unless given):
  * one ``torch.Generator`` seeded per workload; fp32 ``randn`` for Q, then K,
    then V (V multiplied by ``v_std``), all in [B, S, H, D] order;
  * activation-like workloads then draw, per KV head, 4 distinct channel
    indices (``randperm(D)[:4]``), multiply those channels by 20 in K and in
    every query head of the group, and apply half-split RoPE with
    theta = 1e6 at positions 0..S-1 to Q and K;
  * finally Q, K, V are rounded to bfloat16 ("generated in BF16").
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    Dqk: int
    Dv: int
    seed: int = 0
    v_std: float = 1.0
    outliers: int = 0          # outlier channels per KV head (activation-like)
    outlier_gain: float = 20.0
    rope_theta: Optional[float] = None
    description: str = ""

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.Dqk)

    @property
    def causal_flops(self) -> float:
        """B*Hq*S^2*(Dqk+Dv): the causal FLOP count the benchmark reports."""
        return float(self.B) * self.Hq * self.S * self.S * (self.Dqk + self.Dv)

    def with_seq(self, S: int, name: Optional[str] = None) -> "Workload":
        return dataclasses.replace(self, S=S, name=name or f"{self.name}_S{S}")


# The five workloads of the benchmark plan (names describe shape, not order).
WORKLOADS: Dict[str, Workload] = {
    "gauss_b1_h2_s1k_d128": Workload(
        "gauss_b1_h2_s1k_d128", B=1, Hq=2, Hkv=2, S=1024, Dqk=128, Dv=128,
        description="small Gaussian case, MHA, 1K tokens"),
    "gauss_b2_gqa32x8_s8k_d128": Workload(
        "gauss_b2_gqa32x8_s8k_d128", B=2, Hq=32, Hkv=8, S=8192, Dqk=128, Dv=128,
        description="Gaussian GQA, batch 2, 8K tokens"),
    "gauss_b1_gqa32x8_s32k_d128": Workload(
        "gauss_b1_gqa32x8_s32k_d128", B=1, Hq=32, Hkv=8, S=32768, Dqk=128, Dv=128,
        description="kernel-benchmark shape: Gaussian GQA, 32K tokens"),
    "gauss_b1_mla16_s32k_d192": Workload(
        "gauss_b1_mla16_s32k_d192", B=1, Hq=16, Hkv=16, S=32768, Dqk=192, Dv=128,
        description="MLA prefill head shape, Gaussian, 32K tokens"),
    "act_b1_gqa32x8_s16k_d128": Workload(
        "act_b1_gqa32x8_s16k_d128", B=1, Hq=32, Hkv=8, S=16384, Dqk=128, Dv=128,
        v_std=0.5, outliers=4, outlier_gain=20.0, rope_theta=1.0e6,
        description="activation-like: outlier channels x20 + RoPE(1e6), V~N(0,0.5^2)"),
}

SMALL = "gauss_b1_h2_s1k_d128"
BENCH = "gauss_b1_gqa32x8_s32k_d128"


def get(name: str) -> Workload:
    return WORKLOADS[name]


def custom(B: int, Hq: int, Hkv: int, S: int, Dqk: int = 128, Dv: int = 128,
           seed: int = 0, **kw) -> Workload:
    name = kw.pop("name", f"custom_b{B}_h{Hq}x{Hkv}_s{S}_d{Dqk}x{Dv}_seed{seed}")
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, S=S, Dqk=Dqk, Dv=Dv, seed=seed, **kw)


def _rope_half_split(x: torch.Tensor, theta: float) -> torch.Tensor:
    """Rotary position embedding, half-split convention, positions 0..S-1.

    x: fp32 [B, S, H, D]. Angles are formed in float64 and applied in fp32.
    """
    B, S, H, D = x.shape
    half = D // 2
    inv_freq = theta ** (-torch.arange(0, half, dtype=torch.float64) * 2.0 / D)
    ang = torch.arange(S, dtype=torch.float64)[:, None] * inv_freq[None, :]
    cos = torch.cos(ang).to(torch.float32)[None, :, None, :]
    sin = torch.sin(ang).to(torch.float32)[None, :, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def make_qkv(w: Workload, device: str = "cpu"):
    """Return (q, k, v) bf16 tensors of shape [B,S,Hq,Dqk], [B,S,Hkv,Dqk], [B,S,Hkv,Dv].

    Drawn on the CPU from the workload's seed so that every consumer sees the
    same values; moved to ``device`` at the end.
    """
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    q = torch.randn((w.B, w.S, w.Hq, w.Dqk), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.S, w.Hkv, w.Dqk), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.S, w.Hkv, w.Dv), generator=g, dtype=torch.float32)
    if w.v_std != 1.0:
        v.mul_(w.v_std)
    if w.outliers:
        group = w.Hq // w.Hkv
        for hk in range(w.Hkv):
            chans = torch.randperm(w.Dqk, generator=g)[: w.outliers]
            k[:, :, hk, chans] *= w.outlier_gain
            for hq in range(hk * group, (hk + 1) * group):
                q[:, :, hq, chans] *= w.outlier_gain
    if w.rope_theta is not None:
        q = _rope_half_split(q, w.rope_theta)
        k = _rope_half_split(k, w.rope_theta)
    q = q.to(torch.bfloat16)
    k = k.to(torch.bfloat16)
    v = v.to(torch.bfloat16)
    if device != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v


def sample_rows(S: int, n: int = 256, seed: int = 1, tile: int = 128) -> List[int]:
    """Query rows for sampled checks: first/last rows and every tile edge that
    fits, then seeded random rows, sorted and unique."""
    rows = {0, S - 1}
    for t in range(0, S, tile):
        for r in (t, t + 1, t + tile - 1):
            if r < S and len(rows) < n // 2:
                rows.add(r)
    g = torch.Generator(device="cpu").manual_seed(seed)
    while len(rows) < min(n, S):
        rows.add(int(torch.randint(0, S, (1,), generator=g)))
    return sorted(rows)
