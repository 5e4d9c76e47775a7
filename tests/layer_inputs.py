"""Test helper: one MoE layer's inputs on both sides.

The seeded fp32 draws come from ``block_scaled_mx_gb300.workload``; the GPU side
quantises them with the library (``mx_quantize_weights``), the oracle side with
the oracle's own quantiser, from the same fp32 values.  Nothing computed by the
CUDA path is handed to the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from block_scaled_mx_gb300 import mxmoe as mx
from block_scaled_mx_gb300 import workload as W


class Layer:
    pass


def build_layer(wl: W.Workload, seed: int = 0, device="cuda", oracle_experts="all", draw_device=None):
    """Returns a Layer with GPU tensors (logits, x, canonical MX weights, prepared
    MoELayer) and, for the experts in `oracle_experts` ("all", "none" or a set),
    the oracle-quantised weights."""
    draw_device = draw_device or device
    fmt = mx.FORMATS[wl.fmt]
    E1 = wl.E + 1
    cdiv = 1 if fmt == mx.MX_E4M3 else 2
    L = Layer()
    L.wl, L.fmt = wl, fmt
    logits, x = W.draw_router_and_activations(wl, seed, draw_device)
    L.logits, L.x = logits.to(device), x.to(device)
    L.logits_np = logits.cpu().numpy()
    L.x_bits = W.bf16_bits(x)
    L.w1c = torch.empty(E1, 2 * wl.I, wl.H // cdiv, dtype=torch.uint8, device=device)
    L.w1s = torch.empty(E1, 2 * wl.I, wl.H // 32, dtype=torch.uint8, device=device)
    L.w2c = torch.empty(E1, wl.H, wl.I // cdiv, dtype=torch.uint8, device=device)
    L.w2s = torch.empty(E1, wl.H, wl.I // 32, dtype=torch.uint8, device=device)
    L.o1c, L.o1s, L.o2c, L.o2s = [None] * E1, [None] * E1, [None] * E1, [None] * E1
    for e in range(E1):
        w1, w2 = W.draw_expert_weights(wl, e, seed, draw_device)
        w1d, w2d = w1.to(device), w2.to(device)
        mx.mx_quantize_weights(w1d, fmt, L.w1c[e], L.w1s[e])
        mx.mx_quantize_weights(w2d, fmt, L.w2c[e], L.w2s[e])
        if oracle_experts == "all" or (oracle_experts != "none" and e in oracle_experts):
            L.o1c[e], L.o1s[e] = oracle.quantize_f32(w1.cpu().numpy(), fmt)
            L.o2c[e], L.o2s[e] = oracle.quantize_f32(w2.cpu().numpy(), fmt)
        del w1, w2, w1d, w2d
    L.layer = mx.MoELayer(L.w1c, L.w1s, L.w2c, L.w2s, fmt, wl.H, wl.I, wl.E, wl.k)
    return L


def oracle_forward(L: Layer, tokens=None, want_h=False):
    wl = L.wl
    return oracle.moe_forward(L.x_bits, L.logits_np, wl.k, L.o1c, L.o1s, L.o2c, L.o2s, L.fmt, wl.I,
                              tokens=tokens, want_h=want_h)


def out_errors(got: np.ndarray, ref: np.ndarray):
    """(relative L2 error, max-abs error / RMS of the reference)."""
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return rel, float(np.max(np.abs(got - ref)) / max(rms, 1e-300))


# tolerance on the layer output: relative L2 error and max-abs error over the
# oracle output's RMS (fp32 tensor-core accumulation and fp32 SwiGLU against the
# fp64 oracle)
OUT_REL_L2 = 5e-3
OUT_MAX_ABS_OVER_RMS = 0.03
