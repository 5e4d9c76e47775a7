#!/usr/bin/env python3
"""Benchmark of the MX block-scaled MoE expert layer on GB300.

One step = one pass of the whole layer (activation quantisation, top-k
routing, permutation, grouped gate/up GEMM + SwiGLU + requant, grouped down
GEMM + combine) over one batch of a synthetic workload, on one GPU.  The
headline workload is the decode MXFP8 layer (T=32, H=4096, I=1536, 128 experts
top-8 + 1 shared); the same run measures the other four layer shapes and puts
them under "workloads" in the same JSON line (rank 0 prints one line).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--only] [--impl reference] [--no-cpu-baseline]

--impl reference times the CPU oracle (plain C, fp64) on the same workload,
each step one oracle call on a batch of its tokens (the whole batch when K of
them fit the time budget).  For N > 1 (torchrun) every rank runs an independent
replica of the layer ("replicas only": the layer does not shard across GPUs
here); throughput is the sum over ranks at the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_scaled_mx_gb300 import workload as W  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
MX8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 vs 2.25 PFLOP/s)
METRIC = "MoE layer tokens/s"
# the headline first, then the other layer shapes
WORKLOAD_ORDER = ["decode_mxfp8", "tiny", "specverify_mxfp4", "decode_mxfp4", "prefill_mxfp8"]


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode_mxfp8", choices=list(W.WORKLOADS))
    ap.add_argument("--only", action="store_true", help="measure the --workload shape alone")
    ap.add_argument("--impl", default="mxmoe", choices=["mxmoe", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0,
                    help="oracle time per workload for the GPU arm's cpu_baseline")
    ap.add_argument("--reference-budget-s", type=float, default=180.0,
                    help="oracle time of the whole --impl reference run")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    src = "fallback"
    hbm, bf16, bf16s = FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = float(d.get("hbm_gbs", hbm))
            bf16 = float(d.get("bf16_tflops", bf16))
            bf16s = float(d.get("bf16_tflops_sustained", bf16s))
            src = "measured"
        except Exception:
            pass
    return {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_tflops_sustained": bf16s, "source": src}


def config_of(wl: W.Workload, world: int) -> dict:
    """The workload description both arms print (identical keys and values)."""
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k, "shared_experts": 1,
            "weights": "MXFP8 E4M3" if wl.fmt == "e4m3" else "MXFP4 E2M1", "activations": "MXFP8 E4M3",
            "router_bias": "1.1*ln(1/(e+1))" if wl.zipf_bias else "none",
            "l2": "flushed between steps (2x L2 write outside the timed events)",
            "parallelism": f"replicas x{world}"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    PERIOD_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []          # (arrival time, csv line)
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, t0: float, t1: float):
        """The timed region, in perf_counter seconds: only samples taken inside it
        (or, when it is shorter than one period, the ones next to it) count."""
        self.window = (t0, t1)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, window=None):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        window = window or self.window
        if window is not None:
            t0, t1 = window
            pad = 1.5 * self.PERIOD_MS * 1e-3
            inside = [ln for t, ln in lines if t0 <= t <= t1 + pad]
            lines = inside or [ln for t, ln in lines if t0 - pad <= t <= t1 + 2 * pad]
        else:
            lines = [ln for _, ln in lines]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ layer setup
def build_gpu_layer(wl: W.Workload, dev):
    from block_scaled_mx_gb300 import mxmoe as mx

    fmt = mx.FORMATS[wl.fmt]
    E1 = wl.E + 1
    cdiv = 1 if fmt == mx.MX_E4M3 else 2
    logits, x = W.draw_router_and_activations(wl, 0, dev)
    w1c = torch.empty(E1, 2 * wl.I, wl.H // cdiv, dtype=torch.uint8, device=dev)
    w1s = torch.empty(E1, 2 * wl.I, wl.H // 32, dtype=torch.uint8, device=dev)
    w2c = torch.empty(E1, wl.H, wl.I // cdiv, dtype=torch.uint8, device=dev)
    w2s = torch.empty(E1, wl.H, wl.I // 32, dtype=torch.uint8, device=dev)
    for e in range(E1):
        w1, w2 = W.draw_expert_weights(wl, e, 0, dev)
        mx.mx_quantize_weights(w1, fmt, w1c[e], w1s[e])
        mx.mx_quantize_weights(w2, fmt, w2c[e], w2s[e])
        del w1, w2
    layer = mx.MoELayer(w1c, w1s, w2c, w2s, fmt, wl.H, wl.I, wl.E, wl.k)
    del w1c, w1s, w2c, w2s
    torch.cuda.synchronize()
    return layer, logits, x


def weight_bytes_per_expert(wl: W.Workload):
    elem = 1.0 if wl.fmt == "e4m3" else 0.5
    w1 = 2 * wl.I * wl.H * elem + 2 * wl.I * wl.H / 32
    w2 = wl.H * wl.I * elem + wl.H * wl.I / 32
    return w1, w2


def gateup_algorithmic_bytes(wl: W.Workload, touched: int) -> float:
    """Bytes the gate/up GEMM must move at least: the touched experts' W1 codes
    and scales, each token's MXFP8 activation row once, h written once."""
    w1b, _ = weight_bytes_per_expert(wl)
    mx8 = 1.0 + 1.0 / 32
    return touched * w1b + wl.T * wl.H * mx8 + wl.slots * wl.I * mx8


def source_hash():
    """Hash of the code (comments and blank lines dropped) of the sources the
    dominant kernel and its launch schedule are built from."""
    import re

    h = hashlib.sha256()
    for f in ("gemm.cu", "ptx.cuh", "common.cuh", "api.cu"):
        text = open(os.path.join(ROOT, "block_scaled_mx_gb300", "csrc", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_tag: str, wl_name: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"ncu_{kernel_tag}_{wl_name}.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        if d.get("source_hash") != source_hash():
            return None
        return float(d["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ CPU oracle timing
_ORACLE_WEIGHTS = {}   # (H, I, E, fmt, seed, expert) -> oracle-quantised W1/W2 codes and scales


class OracleRunner:
    """The CPU oracle on a workload: each call evaluates a batch of its tokens
    (the experts those tokens touch are drawn and quantised by the oracle on
    first use, untimed; workloads with the same weight shapes and format share
    them)."""

    def __init__(self, wl: W.Workload):
        import oracle

        oracle.build()
        self.oracle, self.wl = oracle, wl
        logits, x = W.draw_router_and_activations(wl, 0, "cpu")
        self.ids, _ = oracle.route_topk(logits.numpy(), wl.k)
        self.fmt = oracle.E4M3 if wl.fmt == "e4m3" else oracle.E2M1
        self.w = [[None] * (wl.E + 1) for _ in range(4)]
        self.x_bits, self.lg = W.bf16_bits(x), logits.numpy()
        self.next_token = 0
        self.threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))

    def tokens(self, n: int):
        toks = sorted(set((self.next_token + i) % self.wl.T for i in range(n)))
        self.next_token += n
        return toks

    def prepare(self, toks):
        wl = self.wl
        for e in set(int(e) for e in self.ids[toks].ravel()) | {wl.E}:
            if self.w[0][e] is not None:
                continue
            key = (wl.H, wl.I, wl.E, wl.fmt, 0, e)
            if key not in _ORACLE_WEIGHTS:
                w1, w2 = W.draw_expert_weights(wl, e, 0, "cpu")
                _ORACLE_WEIGHTS[key] = (*self.oracle.quantize_f32(w1.numpy(), self.fmt),
                                        *self.oracle.quantize_f32(w2.numpy(), self.fmt))
            for i in range(4):
                self.w[i][e] = _ORACLE_WEIGHTS[key][i]

    def call(self, toks):
        """Seconds of one oracle call on the token list `toks` (weights prepared first, untimed)."""
        self.prepare(toks)
        t0 = time.perf_counter()
        self.oracle.moe_forward(self.x_bits, self.lg, self.wl.k, *self.w, self.fmt, self.wl.I,
                                tokens=None if len(toks) == self.wl.T else toks)
        return time.perf_counter() - t0

    def baseline(self, budget_s: float, n_tokens: int, one_core: bool = False):
        """cpu_baseline entry: oracle calls on batches of n_tokens until budget_s
        of oracle time is spent (at least one call)."""
        done, spent, calls = 0, 0.0, 0
        while calls == 0 or (spent < budget_s and calls < 64):
            toks = self.tokens(n_tokens)
            spent += self.call(toks)
            done, calls = done + len(toks), calls + 1
        what = "the whole batch" if n_tokens >= self.wl.T else f"{n_tokens} of its {self.wl.T} tokens"
        sample = (f"{calls} oracle call(s), each on {what} of the {self.wl.name} workload "
                  f"({done} tokens in {spent:.1f} s; each call decodes the touched experts' weights to fp64 "
                  f"and runs fp64 loops)")
        d = {"value": done / spent, "unit": "tokens/s", "cores": 1 if one_core else self.threads, "kind": "oracle",
             "sample": sample}
        return d


# ------------------------------------------------------------------ replicas
def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank gets the maximum of ``ms`` over the
    process group (a tensor on ``device``: the GPU under NCCL, the CPU under gloo)."""
    if world <= 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, T: int, ms: float) -> float:
    """Tokens/s of the whole job: each of ``world`` replicas runs the layer on
    its own T tokens, and the job takes as long as the slowest one (``ms``)."""
    return world * T / (ms * 1e-3)


def cpu_sample_tokens(wl: W.Workload) -> int:
    """Tokens per oracle call for the GPU arm's cpu_baseline: the whole batch,
    except the 8192-token prefill (minutes of fp64 work), which takes a sample."""
    return wl.T if wl.T <= 256 else 8


# ------------------------------------------------------------------ reference arm
def reference_plan(t_first: float, n_first: int, runner: OracleRunner, steps: int, budget_s: float):
    """Tokens per step: the whole batch when `steps` whole-batch calls fit the
    budget, else the largest batch whose estimated call time (the first call's
    time scaled by the experts it touches) fits."""
    wl = runner.wl
    if steps * t_first <= budget_s:
        return n_first
    touched_full = len(set(int(e) for e in runner.ids[:n_first].ravel()) | {wl.E})
    n = n_first
    while n > 1:
        n = max(1, n // 2)
        touched = len(set(int(e) for e in runner.ids[:n].ravel()) | {wl.E})
        if steps * t_first * touched / touched_full <= budget_s:
            break
    return n


def run_reference(args, wl, rank, world):
    if rank != 0:
        return
    runner = OracleRunner(wl)
    # the first warm-up step (untimed) is a call on the whole batch, or on the
    # prefill sample: its time sizes the steps
    n0 = cpu_sample_tokens(wl)
    t_first = runner.call(list(range(n0)))
    n_step = reference_plan(t_first, n0, runner, args.steps, args.reference_budget_s)
    for _ in range(max(0, args.warmup - 1)):
        runner.call(runner.tokens(n_step))
    times, done = [], 0
    for _ in range(args.steps):
        toks = runner.tokens(n_step)
        times.append(runner.call(toks))
        done += len(toks)
    spent = float(np.sum(times))
    rate = done / spent
    what = "the whole batch" if n_step >= wl.T else f"{n_step} of its {wl.T} tokens (taken in turn)"
    sample = (f"each step one oracle call on {what} of the {wl.name} workload; "
              f"{args.steps} timed steps after {args.warmup} warm-up, {spent:.1f} s of oracle time")
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * spent / args.steps, "tokens_per_step": n_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, world),
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": runner.threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def time_fused(layer, x, logits, out, steps, warmup, flush, stream, dev, opts=None):
    """Mean us of moe_forward (or moe_forward_ex with `opts`) replayed from a
    CUDA graph, L2 flushed between steps outside the events."""
    for _ in range(warmup):
        layer.forward(x, logits, out, opts=opts)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            layer.forward(x, logits, out, opts=opts)
    stream.wait_stream(cap)
    for _ in range(warmup):
        flush.fill_(1)
        graph.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.fill_(1)
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return 1e3 * float(np.mean([a.elapsed_time(b) for a, b in ev]))


def measure_variants(args, layer, wl, x, logits, flush, stream, dev, folded_us, touched):
    """The layer variants timed beside the default: the shared expert as its own
    dense launches (the A/B of the folded table), the SwiGLU-OAI epilogue, the
    router GEMM, and (MXFP4 weights) MXFP4 activations on the packed-FP4 MMA."""
    from block_scaled_mx_gb300 import mxmoe as mx

    out = torch.empty(wl.T, wl.H, dtype=torch.float32, device=dev)
    dense = mx.layer_opts(shared="dense")
    oai = mx.layer_opts("swiglu_oai", alpha=1.702, limit=7.0)
    dense_us = time_fused(layer, x, logits, out, args.steps, args.warmup, flush, stream, dev, dense)
    oai_us = time_fused(layer, x, logits, out, args.steps, args.warmup, flush, stream, dev, oai)
    if mx.moe_get_status(layer.workspace(wl.T)):
        raise RuntimeError(f"{wl.name}: device status error in a layer variant")
    # the router GEMM with top-k in its epilogue, on this workload's T, H, E, k
    g = torch.Generator(device=dev).manual_seed(7)
    w_r = (torch.randn(wl.E, wl.H, generator=g, device=dev) / wl.H ** 0.5).to(torch.bfloat16)
    ids = torch.empty(wl.T, wl.k, dtype=torch.int32, device=dev)
    tw = torch.empty(wl.T, wl.k, dtype=torch.float32, device=dev)
    # room for the logits: batches of up to 128 tokens then take the small-batch kernel
    rws = mx.alloc_workspace(256 + 4 * wl.T * wl.E, dev)
    for _ in range(args.warmup):
        mx.moe_route_gemm_topk(x, w_r, wl.k, rws, topk_ids=ids, topk_w=tw)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            mx.moe_route_gemm_topk(x, w_r, wl.k, rws, topk_ids=ids, topk_w=tw)
    stream.wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(1)
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if mx.moe_get_status(rws):
        raise RuntimeError(f"{wl.name}: device status error in the router GEMM")
    router_us = 1e3 * float(np.mean([a.elapsed_time(b) for a, b in ev]))
    router = {"us": router_us, "tflops": 2.0 * wl.T * wl.H * wl.E / (router_us * 1e-6) / 1e12,
              "gbs": (wl.E * wl.H * 2 + wl.T * wl.H * 2 + wl.T * wl.k * 8) / (router_us * 1e-6) / 1e9,
              "launches": 1, "timing": "CUDA graph of the call, CUDA events, L2 flushed"}
    res = {}
    if wl.fmt == "e2m1":
        # MXFP4 activations and h: both grouped GEMMs on the packed-FP4 MMA
        # (changes the numerics: its own oracle path and tolerance in the tests)
        a4 = mx.layer_opts(act_fmt="e2m1")
        a4_us = time_fused(layer, x, logits, out, args.steps, args.warmup, flush, stream, dev, a4)
        if mx.moe_get_status(layer.workspace(wl.T)):
            raise RuntimeError(f"{wl.name}: device status error in the MXFP4-activation layer")
        w1b, w2b = weight_bytes_per_expert(wl)
        res["mxfp4_activations"] = {
            "us_per_layer": a4_us, "speedup_vs_mxfp8_activations": folded_us / a4_us,
            "layer_roofline_frac": touched * (w1b + w2b) / (a4_us * 1e-6) / 1e9 / peaks()["hbm_gbs"],
            "mma": "tcgen05 kind::mxf4 block_scale scale_vec::2X"}
    return {**res, "router_gemm_topk": router,
            "shared_expert": {"folded_us": folded_us, "dense_us": dense_us,
                              "folded_speedup": dense_us / folded_us,
                              "dense_launches": mx.moe_forward_launches_ex(wl.T, wl.H, wl.I, wl.E, wl.k, layer.fmt, dense)},
            "swiglu_oai": {"us_per_layer": oai_us, "alpha": 1.702, "limit": 7.0}}


def measure_workload(args, wl, dev, world, clk, with_cpu):
    """Times one workload; returns its entry (headline keys included)."""
    from block_scaled_mx_gb300 import mxmoe as mx

    layer, logits, x = build_gpu_layer(wl, dev)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    fmt = layer.fmt
    stream = torch.cuda.current_stream()
    # step-call buffers
    act_c = torch.empty(T, H, dtype=torch.uint8, device=dev)
    act_s = torch.empty(T, H // 32, dtype=torch.uint8, device=dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    tw = torch.empty(T, k, dtype=torch.float32, device=dev)
    counts = torch.empty(E + 1, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 2, dtype=torch.int32, device=dev)
    ss = torch.empty(T * (k + 1), dtype=torch.int32, device=dev)
    pws = mx.alloc_workspace(mx.moe_permute_workspace_size(T, E, k), dev)
    gws = mx.alloc_workspace(mx.moe_gemm_workspace_size(T, H, I, E, k), dev)
    h_c = torch.empty(T * (k + 1), I, dtype=torch.uint8, device=dev)
    h_s = torch.empty(T * (k + 1), I // 32, dtype=torch.uint8, device=dev)
    out = torch.empty(T, H, dtype=torch.float32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    def step(ev):
        ev[0].record(stream)
        mx.mx_quantize_act(x, act_c, act_s)
        ev[1].record(stream)
        mx.moe_route_topk(logits, k, ids, tw)
        ev[2].record(stream)
        mx.moe_permute(ids, E, counts, offsets, ss, pws)
        out.zero_()
        ev[3].record(stream)
        mx.moe_grouped_gemm_swiglu(act_c, act_s, offsets, ss, layer.w1, fmt, T, H, I, E, k, h_c, h_s, gws)
        ev[4].record(stream)
        mx.moe_grouped_gemm_down_combine(h_c, h_s, offsets, ss, tw, layer.w2, fmt, T, H, I, E, k, out, gws)
        ev[5].record(stream)

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(6)]  # noqa: E731
    for _ in range(args.warmup):
        flush.fill_(1)
        step(mk())
    torch.cuda.synchronize()
    if mx.moe_get_status(pws) or mx.moe_get_status(gws):
        raise RuntimeError(f"{wl.name}: device status error during warm-up")
    cnt = counts.cpu().numpy()
    touched = int(np.count_nonzero(cnt))
    w1b, w2b = weight_bytes_per_expert(wl)
    evs = [mk() for _ in range(args.steps)]
    out_f = torch.empty(T, H, dtype=torch.float32, device=dev)
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for _ in range(args.warmup):
        flush.fill_(1)
        layer.forward(x, logits, out_f)
    torch.cuda.synchronize()
    # The fused call is replayed from a CUDA graph in the timed loop: the host
    # then enqueues one graph launch per step, so a slow or busy host cannot
    # leave the GPU idle between the timed events (same kernels, same launch
    # attributes, captured from the public call).
    fused_mode = "cuda graph of moe_forward"
    try:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                layer.forward(x, logits, out_f)
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize()
        run_fused = graph.replay
    except Exception:  # capture unavailable: time the eager call
        fused_mode = "moe_forward (eager)"
        run_fused = lambda: layer.forward(x, logits, out_f)  # noqa: E731
    for _ in range(args.warmup):
        flush.fill_(1)
        run_fused()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        # (a) the layer through the fused single call: the step time
        flush.fill_(1)          # L2 flush, outside the timed events
        fev[i][0].record(stream)
        run_fused()
        fev[i][1].record(stream)
        # (b) the same kernels through the step-wise calls, events between
        #     them: per-kernel durations for the roofline
        flush.fill_(1)
        step(evs[i])
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    if world > 1:
        torch.distributed.barrier()
    per = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(5)] for i in range(args.steps)])
    fused_ms = np.array([a.elapsed_time(b) for a, b in fev])
    ms = max_over_ranks(float(fused_ms.mean()), world, dev)
    value = replica_throughput(world, T, ms)

    # ---- e2e through the public single call with host buffers: x and the
    #      router logits sit in one pinned staging buffer (one host-to-device
    #      copy a step), the output comes back in a second
    xb, lb = T * H * 2, T * E * 4
    in_h = torch.empty(xb + lb, dtype=torch.uint8).pin_memory()
    in_h[:xb].copy_(x.cpu().contiguous().view(torch.uint8).reshape(-1))
    in_h[xb:].copy_(logits.cpu().contiguous().view(torch.uint8).reshape(-1))
    out_h = torch.empty(T, H, dtype=torch.float32).pin_memory()
    in_d = torch.empty(xb + lb, dtype=torch.uint8, device=dev)
    x_d = in_d[:xb].view(torch.bfloat16).view(T, H)
    lg_d = in_d[xb:].view(torch.float32).view(T, E)
    out_d = torch.empty(T, H, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        in_d.copy_(in_h, non_blocking=True)
        layer.forward(x_d, lg_d, out_d)
        out_h.copy_(out_d, non_blocking=True)
    torch.cuda.synchronize()
    # the staged inputs are the device inputs (the combine's fp32 atomics may
    # add in another order)
    ref_out = layer.forward(x, logits).cpu()
    if not torch.allclose(out_h, ref_out, rtol=0, atol=1e-5 * float(ref_out.abs().max()) + 1e-30):
        raise RuntimeError(f"{wl.name}: end-to-end output differs from the device-input call")
    e2e_ms = []
    for i in range(args.steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        in_d.copy_(in_h, non_blocking=True)
        layer.forward(x_d, lg_d, out_d)
        out_h.copy_(out_d, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e = max_over_ranks(float(np.mean(e2e_ms)), world, dev)

    # ---- the grouped-GEMM kernels alone: the step-wise calls again, with the
    #      library recording CUDA events around each GEMM launch on its stream
    #      (the wide schedule's gate/up call also runs the row gather, which
    #      the call's own events include)
    mx.mx_debug_time_gemms(True)
    for i in range(args.steps):
        flush.fill_(1)
        step(mk())
    torch.cuda.synchronize()
    k_ms, k_epi = mx.mx_debug_gemm_times()
    mx.mx_debug_time_gemms(False)
    g1k = [t for t, e in zip(k_ms, k_epi) if e == 0]
    g2k = [t for t, e in zip(k_ms, k_epi) if e == 1]
    if mx.moe_get_status(layer.workspace(T)):
        raise RuntimeError(f"{wl.name}: device status error in moe_forward")
    variants = measure_variants(args, layer, wl, x, logits, flush, stream, dev, ms * 1e3, touched)

    pk = peaks()
    gemm1_ms = float(per[:, 3].mean())
    gemm2_ms = float(per[:, 4].mean())
    g1_kernel_ms = float(np.mean(g1k)) if g1k else gemm1_ms
    g2_kernel_ms = float(np.mean(g2k)) if g2k else gemm2_ms
    slots = T * (k + 1)
    flops = 6.0 * slots * H * I
    tc_peak = pk["bf16_tflops"] * MX8_OVER_BF16
    hbm_peak = pk["hbm_gbs"]
    bw = touched * (w1b + w2b)
    layer_floor_ms = max(flops / (tc_peak * 1e12), bw / (hbm_peak * 1e9)) * 1e3
    dominant_hbm = flops / (tc_peak * 1e12) < bw / (hbm_peak * 1e9)
    kname = "k_grouped_gemm (gate/up + SwiGLU + requant)"
    if dominant_hbm:
        g1_bytes = gateup_algorithmic_bytes(wl, touched)
        achieved = g1_bytes / (g1_kernel_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "traffic": ncu_traffic("gemm1", wl.name), "kernel": kname, "algorithmic_bytes": g1_bytes,
                "kernel_ms": g1_kernel_ms, "peak_source": pk["source"] + " copy bandwidth (burst)"}
    else:
        g1_flops = 4.0 * slots * H * I
        achieved = g1_flops / (g1_kernel_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": achieved / tc_peak, "traffic": ncu_traffic("gemm1", wl.name), "kernel": kname,
                "algorithmic_flops": g1_flops, "kernel_ms": g1_kernel_ms,
                "peak_source": pk["source"] + " bf16 burst x2 (nominal MXFP8/bf16 ratio)"}
    fused_launches = mx.moe_forward_launches(T, H, I, E, k, fmt)
    nperm = 1 if T <= 256 else 2
    wide = fused_launches > 3 and (T * (k + 1)) / (E + 1) >= 48
    step_launches = 1 + 1 + nperm + (2 if wide else 1) + 1
    entry = {
        "us_per_layer": ms * 1e3, "tokens_s": value, "ms_per_step": ms, "steps": args.steps, "warmup": args.warmup,
        "launches_per_layer": fused_launches,
        "timing": f"value: {fused_mode}; kernels_ms: the step-wise calls in the same loop (CUDA events between "
                  "calls); *_kernel and roofline.kernel_ms: a second pass of the step-wise calls with CUDA events the "
                  "library records around each grouped-GEMM launch",
        "roofline": roof,
        "layer_roofline": {"floor_us": layer_floor_ms * 1e3, "frac": layer_floor_ms / ms,
                           "touched_experts": touched, "weight_bytes": bw, "flops": flops,
                           "bound": "hbm" if dominant_hbm else "tensor"},
        "kernels_ms": {"quantize": float(per[:, 0].mean()), "topk": float(per[:, 1].mean()),
                       "permute+zero": float(per[:, 2].mean()), "gateup_call": gemm1_ms, "down_call": gemm2_ms,
                       "gateup_kernel": g1_kernel_ms, "down_kernel": g2_kernel_ms,
                       "step_calls_total": float(per.sum(1).mean())},
        "e2e": {"value": replica_throughput(world, T, e2e), "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2 + T * E * 4,
                "d2h_bytes_per_step": T * H * 4, "ms_per_step": e2e},
        "clocks": clk.summary((t_wall0, t_wall1)),
        "gpu_launches": (fused_launches + step_launches) * args.steps,
        "wall_s_timed": t_wall1 - t_wall0,
        "variants": variants,
    }
    del layer, flush
    torch.cuda.empty_cache()
    if with_cpu:
        entry["cpu_baseline"] = cpu_baseline(args, wl)
    return entry


def cpu_baseline(args, wl):
    try:
        runner = OracleRunner(wl)
        cpu = runner.baseline(args.cpu_budget_s, cpu_sample_tokens(wl))
        if wl.T <= 16:  # the smallest configurations: also one core, the oracle's per-core speed
            try:
                runner.oracle.set_threads(1)
                one = runner.baseline(args.cpu_budget_s / 3, cpu_sample_tokens(wl), one_core=True)
            finally:
                runner.oracle.set_threads(0)
            cpu["value_1core"] = one["value"]
            cpu["sample_1core"] = one["sample"]
        return cpu
    except Exception as exc:  # the GPU number stands without it
        return {"value": None, "unit": "tokens/s", "cores": None, "kind": "oracle", "sample": f"failed: {exc}"}


def run_gpu(args, rank, world, local):
    from block_scaled_mx_gb300 import build as B
    from block_scaled_mx_gb300 import mxmoe as mx

    if rank == 0 or world == 1:
        B.build()
    if world > 1:
        torch.distributed.barrier()
        B.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    with_cpu = world == 1 and not args.no_cpu_baseline
    names = [args.workload] + ([] if args.only else [n for n in WORKLOAD_ORDER if n != args.workload])
    entries = {}
    with ClockSampler(local) as clk:
        time.sleep(0.3)             # the sampler's first lines arrive before the first timed region
        for n in names:
            entries[n] = measure_workload(args, W.WORKLOADS[n], dev, world, clk, with_cpu and rank == 0)
        time.sleep(3 * ClockSampler.PERIOD_MS * 1e-3)
    if rank != 0:
        return
    head = entries.pop(args.workload)
    wl = W.WORKLOADS[args.workload]
    line = {
        "metric": METRIC, "value": head["tokens_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "us_per_layer": head["us_per_layer"], "launches_per_layer": head["launches_per_layer"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3" if wl.fmt == "e4m3" else "e2m1") + " x e4m3 -> f32 (MX block-scaled)",
        "data": "synthetic",
        "config": config_of(wl, world),
        "timing": head["timing"],
        "roofline": head["roofline"],
        "layer_roofline": head["layer_roofline"],
        "kernels_ms": head["kernels_ms"],
        "e2e": head["e2e"],
        "cpu_baseline": head.get("cpu_baseline"),
        "clocks": head["clocks"],
        "gpu_launches": head["gpu_launches"],
        "wall_s_timed": head["wall_s_timed"],
        "variants": head["variants"],
        "sms": torch.cuda.get_device_properties(dev).multi_processor_count,
        "build": {"stamp": mx.mx_build_stamp(), "compiled_in_this_run": bool(B.LAST_BUILD.get("compiled"))},
        "workloads": {n: dict(e, config=config_of(W.WORKLOADS[n], world)) for n, e in entries.items()},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    wl = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl, rank, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    try:
        run_gpu(args, rank, world, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
