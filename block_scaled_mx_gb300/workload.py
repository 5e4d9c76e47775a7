"""Seeded synthetic inputs for the MX block-scaled sparse-MoE expert layer.

This module only draws numbers; it holds none of the layer's arithmetic (no
quantisation, no routing), so both the CUDA path and the CPU oracle take their
inputs from here.  The five workloads are the layer shapes the benchmark is
quoted on:

  tiny              T=16,   H=256,  I=128,  E=8,   k=2, MXFP8 weights
  decode_mxfp8      T=32,   H=4096, I=1536, E=128, k=8, MXFP8 weights
  decode_mxfp4      T=128,  H=4096, I=1536, E=128, k=8, MXFP4 weights
  prefill_mxfp8     T=8192, H=4096, I=1536, E=128, k=8, MXFP8 weights, Zipf-biased router
  specverify_mxfp4  T=6,    H=2048, I=512,  E=512, k=8, MXFP4 weights

each with one shared expert stored at table index E.  Draw recipe:
  * router logits fp32 [T, E] ~ N(0, 1), then x fp32 [T, H] ~ N(0, 1) rounded
    to bf16 (round-to-nearest-even), both from one generator seeded `seed`;
  * the prefill workload adds 1.1 * ln(1 / (e + 1)) to expert e's logit;
  * expert e (0..E, shared last) draws W1 fp32 [2I, H] (gate rows then up rows)
    and then W2 fp32 [H, I], both N(0, 0.02^2), from its own generator seeded
    `seed * 1000003 + e + 1`, so any single expert can be redrawn on its own.
Generators are torch generators on the requested device; CPU and CUDA streams
differ, so a consumer compares like with like.
"""
from __future__ import annotations


from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    fmt: str            # "e4m3" (MXFP8 weights) or "e2m1" (MXFP4 weights)
    zipf_bias: bool = False

    @property
    def slots(self) -> int:
        return self.T * (self.k + 1)


WORKLOADS = {
    "tiny": Workload("tiny", 16, 256, 128, 8, 2, "e4m3"),
    "decode_mxfp8": Workload("decode_mxfp8", 32, 4096, 1536, 128, 8, "e4m3"),
    "decode_mxfp4": Workload("decode_mxfp4", 128, 4096, 1536, 128, 8, "e2m1"),
    "prefill_mxfp8": Workload("prefill_mxfp8", 8192, 4096, 1536, 128, 8, "e4m3", zipf_bias=True),
    "specverify_mxfp4": Workload("specverify_mxfp4", 6, 2048, 512, 512, 8, "e2m1"),
}

WEIGHT_STD = 0.02


def custom(name: str = "custom", T: int = 16, H: int = 256, I: int = 128, E: int = 8, k: int = 2,
           fmt: str = "e4m3", zipf_bias: bool = False) -> Workload:
    return Workload(name, T, H, I, E, k, fmt, zipf_bias)


def draw_router_and_activations(w: Workload, seed: int = 0, device="cpu"):
    """Returns (logits fp32 [T, E], x bf16 [T, H]) on `device`."""
    g = torch.Generator(device=device).manual_seed(seed)
    logits = torch.randn(w.T, w.E, generator=g, device=device, dtype=torch.float32)
    if w.zipf_bias:
        rank = torch.arange(1, w.E + 1, dtype=torch.float64)
        bias = (1.1 * torch.log(1.0 / rank)).to(torch.float32).to(device)
        logits = logits + bias[None, :]
    x = torch.randn(w.T, w.H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return logits, x


def draw_expert_weights(w: Workload, e: int, seed: int = 0, device="cpu"):
    """Returns (W1 fp32 [2I, H], W2 fp32 [H, I]) of expert e (e == E is shared)."""
    if not 0 <= e <= w.E:
        raise ValueError(f"expert {e} out of range 0..{w.E}")
    g = torch.Generator(device=device).manual_seed(seed * 1000003 + e + 1)
    w1 = torch.randn(2 * w.I, w.H, generator=g, device=device, dtype=torch.float32) * WEIGHT_STD
    w2 = torch.randn(w.H, w.I, generator=g, device=device, dtype=torch.float32) * WEIGHT_STD
    return w1, w2


def expected_touched_experts(w: Workload) -> float:
    """E * (1 - (1 - k/E)^T) + 1: expected experts with at least one token under
    uniform routing, plus the shared expert (bench bookkeeping only)."""
    return w.E * (1.0 - (1.0 - w.k / w.E) ** w.T) + 1.0


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU)."""
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


