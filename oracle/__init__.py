"""CPU oracle for the MX block-scaled sparse-MoE expert layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` may import this package.  The product path
(``block_scaled_mx_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``mx_oracle.c`` (plain C, fp64); this module builds it
with gcc and exposes numpy-level wrappers through ctypes.  Each wrapper cites
the same passage as the C function it calls.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

E4M3 = 0
E2M1 = 1
ACT_SWIGLU = 0
ACT_SWIGLU_OAI = 1


def compile_library(src: str, out: str) -> str:
    """gcc, -O2, OpenMP, no fast-math: ``src`` (C11) -> shared library ``out``."""
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    """Compile ``mx_oracle.c`` into ``liboracle.so``."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_library(_SRC, _LIB_PATH)
    return _LIB_PATH


def _bind(L):
    """Declare the C signatures on a loaded oracle library and return it."""
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int, ctypes.c_int64
    L.orc_decode_e4m3.restype = ctypes.c_double
    L.orc_decode_e4m3.argtypes = [i32]
    L.orc_decode_e2m1.restype = ctypes.c_double
    L.orc_decode_e2m1.argtypes = [i32]
    L.orc_decode_e8m0.restype = ctypes.c_double
    L.orc_decode_e8m0.argtypes = [i32]
    L.orc_quantize_block.argtypes = [P, i32, i32, P, P]
    L.orc_quantize_rows.argtypes = [P, i64, i64, i32, P, P]
    L.orc_quantize_bf16.argtypes = [P, i64, i64, P, P]
    L.orc_quantize_f32.argtypes = [P, i64, i64, i32, P, P]
    L.orc_route_topk.argtypes = [P, i32, i32, i32, P, P]
    L.orc_permute.argtypes = [P, i32, i32, i32, P, P, P]
    L.orc_expert_layer.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, i32, P, i32,
                                   P, P, P, P]
    L.orc_expert_layer_ex.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, i32, P, i32,
                                      P, P, P, P, i32, ctypes.c_double, ctypes.c_double, i32, i32]
    L.orc_router_logits.argtypes = [P, P, i32, i32, i32, P]
    L.orc_route_topk_biased.argtypes = [P, P, i32, i32, i32, P, P]
    L.orc_swiglu_oai.restype = ctypes.c_double
    L.orc_swiglu_oai.argtypes = [ctypes.c_double] * 4
    L.orc_set_threads.argtypes = [i32]
    L.orc_set_threads.restype = None
    return L


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(st: int, what: str):
    if st != 0:
        raise ValueError(f"oracle {what} failed with status {st}")


# ------------------------------------------------------------------ formats
def decode_e4m3(codes) -> np.ndarray:
    """E4M3 code -> value (OCP MX v1.0 element format)."""
    c = np.asarray(codes, dtype=np.int64)
    f = lib().orc_decode_e4m3
    return np.array([f(int(x)) for x in c.ravel()], dtype=np.float64).reshape(c.shape)


def decode_e2m1(codes) -> np.ndarray:
    """E2M1 code (low nibble) -> value (OCP MX v1.0 element format)."""
    c = np.asarray(codes, dtype=np.int64)
    f = lib().orc_decode_e2m1
    return np.array([f(int(x)) for x in c.ravel()], dtype=np.float64).reshape(c.shape)


def decode_e8m0(codes) -> np.ndarray:
    """E8M0 scale code -> 2^(code-127), 0xFF -> NaN (OCP MX v1.0)."""
    c = np.asarray(codes, dtype=np.int64)
    f = lib().orc_decode_e8m0
    return np.array([f(int(x)) for x in c.ravel()], dtype=np.float64).reshape(c.shape)


def quantize_block(v, fmt: int):
    """One block -> (unpacked codes, scale code); shared exponent
    floor(log2(amax)) - emax, RNE, saturate."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    codes = np.zeros(v.size, dtype=np.uint8)
    sc = np.zeros(1, dtype=np.uint8)
    _check(lib().orc_quantize_block(_ptr(v), v.size, fmt, _ptr(codes), _ptr(sc)), "quantize_block")
    return codes, int(sc[0])


def quantize_rows(v, fmt: int):
    """fp64 [rows, K] -> (codes, scales); E2M1 packed two per byte, element 2i low nibble."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows, K = v.shape
    codes = np.zeros((rows, K if fmt == E4M3 else K // 2), dtype=np.uint8)
    scales = np.zeros((rows, K // 32), dtype=np.uint8)
    _check(lib().orc_quantize_rows(_ptr(v), rows, K, fmt, _ptr(codes), _ptr(scales)), "quantize_rows")
    return codes, scales


def quantize_bf16(x_bits: np.ndarray, fmt: int = E4M3):
    """bf16 activations (uint16 bit patterns) [T, H] -> MX codes and scales
    [T, H/32]: MXFP8 codes [T, H], or (fmt = E2M1) MXFP4 codes [T, H/2] packed
    two per byte, element 2i in the low nibble (the bf16 values widened to
    fp64 exactly and quantised by quantize_rows)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    if fmt == E2M1:
        widened = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return quantize_rows(widened, E2M1)
    T, H = x.shape
    codes = np.zeros((T, H), dtype=np.uint8)
    scales = np.zeros((T, H // 32), dtype=np.uint8)
    _check(lib().orc_quantize_bf16(_ptr(x), T, H, _ptr(codes), _ptr(scales)), "quantize_bf16")
    return codes, scales


def quantize_f32(w: np.ndarray, fmt: int):
    """fp32 weights [rows, K] -> MX codes and scales in `fmt`."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, K = w.shape
    codes = np.zeros((rows, K if fmt == E4M3 else K // 2), dtype=np.uint8)
    scales = np.zeros((rows, K // 32), dtype=np.uint8)
    _check(lib().orc_quantize_f32(_ptr(w), rows, K, fmt, _ptr(codes), _ptr(scales)), "quantize_f32")
    return codes, scales


def decode_matrix(codes: np.ndarray, scales: np.ndarray, fmt: int) -> np.ndarray:
    """MX matrix -> fp64 values (code value x 2^(scale-127))."""
    rows = codes.shape[0]
    K = scales.shape[1] * 32
    if fmt == E4M3:
        vals = _E4M3_TABLE()[codes.astype(np.int64)]
    else:
        lo = codes & 0xF
        hi = codes >> 4
        el = np.empty((rows, K), dtype=np.int64)
        el[:, 0::2] = lo
        el[:, 1::2] = hi
        vals = _E2M1_TABLE()[el]
    s = _E8M0_TABLE()[scales.astype(np.int64)]
    return vals * np.repeat(s, 32, axis=1)


_tables = {}


def _E4M3_TABLE():
    if "e4m3" not in _tables:
        _tables["e4m3"] = decode_e4m3(np.arange(256))
    return _tables["e4m3"]


def _E2M1_TABLE():
    if "e2m1" not in _tables:
        _tables["e2m1"] = decode_e2m1(np.arange(16))
    return _tables["e2m1"]


def _E8M0_TABLE():
    if "e8m0" not in _tables:
        _tables["e8m0"] = decode_e8m0(np.arange(256))
    return _tables["e8m0"]


# ------------------------------------------------------------------ router / permute
def route_topk(logits: np.ndarray, k: int):
    """fp32 logits [T, E] -> ids int32 [T, k] (descending logit, lowest index on
    ties), w fp64 [T, k] = softmax over the selected logits."""
    l = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = l.shape
    ids = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    _check(lib().orc_route_topk(_ptr(l), T, E, k, _ptr(ids), _ptr(w)), "route_topk")
    return ids, w


def router_logits(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """bf16 activations [T, H] and bf16 router weights [E, H] (uint16 bit
    patterns) -> fp64 logits [T, E] = x . w^T."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    T, H = x.shape
    E = w.shape[0]
    out = np.zeros((T, E), dtype=np.float64)
    _check(lib().orc_router_logits(_ptr(x), _ptr(w), T, H, E, _ptr(out)), "router_logits")
    return out


def route_topk_biased(logits: np.ndarray, bias: Optional[np.ndarray], k: int):
    """Top-k by the fp32 score logit + bias (lowest index on ties), weights =
    softmax of the chosen experts' unbiased logits; bias None = route_topk."""
    l = np.ascontiguousarray(logits, dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    T, E = l.shape
    ids = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    _check(lib().orc_route_topk_biased(_ptr(l), _ptr(b), T, E, k, _ptr(ids), _ptr(w)), "route_topk_biased")
    return ids, w


def permute(ids: np.ndarray, E: int):
    """ids [T, k] -> counts [E+1], offsets [E+2], sorted_slot [T*(k+1)] (slot id t*(k+1)+j,
    j = k for the shared expert; experts ascending, tokens ascending)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    counts = np.zeros(E + 1, dtype=np.int32)
    offsets = np.zeros(E + 2, dtype=np.int32)
    ss = np.zeros(T * (k + 1), dtype=np.int32)
    _check(lib().orc_permute(_ptr(ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(ss)), "permute")
    return counts, offsets, ss


# ------------------------------------------------------------------ expert layer
def expert_layer(act_codes, act_scales, ids, topk_w, w1c: Sequence, w1s: Sequence, w2c: Sequence,
                 w2s: Sequence, fmt: int, I: int, tokens: Optional[Sequence[int]] = None,
                 want_h: bool = False, want_noq: bool = False, act: int = ACT_SWIGLU, alpha: float = 1.0,
                 limit: float = float("inf"), act_fmt: int = E4M3):
    """Grouped gate/up GEMM + SwiGLU (or SwiGLU-OAI with ``alpha`` and
    ``limit``) + MX requant of h + down GEMM + weighted combine, on already
    quantised activations.  ``act_fmt`` is the activations' MX format; h is
    re-quantised to the same format (MXFP8, or MXFP4 for FP4 activations).
    Weight lists hold E+1 entries (shared expert last); None is allowed for
    experts no requested token uses.

    Returns dict with ``out`` fp64 [n_tokens, H] and optionally ``h_codes`` /
    ``h_scales`` (by slot id) and ``out_noq`` (h not re-quantised)."""
    act_codes = np.ascontiguousarray(act_codes, dtype=np.uint8)
    act_scales = np.ascontiguousarray(act_scales, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    topk_w = np.ascontiguousarray(topk_w, dtype=np.float64)
    T = act_codes.shape[0]
    H = act_scales.shape[1] * 32
    k = ids.shape[1]
    E = len(w1c) - 1
    keep = []

    def arr(lst):
        a = (ctypes.c_void_p * len(lst))()
        for i, x in enumerate(lst):
            if x is None:
                a[i] = None
            else:
                x = np.ascontiguousarray(x, dtype=np.uint8)
                keep.append(x)
                a[i] = x.ctypes.data
        return a

    A1c, A1s, A2c, A2s = arr(w1c), arr(w1s), arr(w2c), arr(w2s)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens), dtype=np.int32)
    n = T if tok is None else tok.size
    out = np.zeros((n, H), dtype=np.float64)
    out_noq = np.zeros((n, H), dtype=np.float64) if want_noq else None
    h_row = I if act_fmt == E4M3 else I // 2
    hc = np.zeros((T * (k + 1), h_row), dtype=np.uint8) if want_h else None
    hs = np.zeros((T * (k + 1), I // 32), dtype=np.uint8) if want_h else None
    st = lib().orc_expert_layer_ex(_ptr(act_codes), _ptr(act_scales), T, H, I, E, k, _ptr(ids), _ptr(topk_w),
                                   ctypes.cast(A1c, ctypes.c_void_p), ctypes.cast(A1s, ctypes.c_void_p),
                                   ctypes.cast(A2c, ctypes.c_void_p), ctypes.cast(A2s, ctypes.c_void_p), fmt,
                                   _ptr(tok), n, _ptr(out), _ptr(out_noq), _ptr(hc), _ptr(hs), int(act),
                                   float(alpha), float(limit), int(act_fmt), int(act_fmt))
    _check(st, "expert_layer")
    res = {"out": out}
    if want_h:
        res["h_codes"], res["h_scales"] = hc, hs
    if want_noq:
        res["out_noq"] = out_noq
    return res


def moe_forward(x_bits, logits, k: int, w1c, w1s, w2c, w2s, fmt: int, I: int, tokens=None, want_h=False,
                want_noq=False, act: int = ACT_SWIGLU, alpha: float = 1.0, limit: float = float("inf"),
                act_fmt: int = E4M3):
    """The whole layer: activation quantisation, routing, permutation (implicit
    in the expert visiting order) and the expert layer."""
    act_codes, act_scales = quantize_bf16(x_bits, act_fmt)
    ids, w = route_topk(logits, k)
    res = expert_layer(act_codes, act_scales, ids, w, w1c, w1s, w2c, w2s, fmt, I, tokens=tokens, want_h=want_h,
                       want_noq=want_noq, act=act, alpha=alpha, limit=limit, act_fmt=act_fmt)
    res.update(act_codes=act_codes, act_scales=act_scales, ids=ids, topk_w=w)
    return res


def swiglu_oai(g, u, alpha: float, limit: float) -> np.ndarray:
    """Elementwise SwiGLU-OAI of the oracle's C code (gate clamped above at
    ``limit``, up to [-limit, limit], g * sigmoid(alpha * g) * (u + 1))."""
    g = np.asarray(g, dtype=np.float64)
    u = np.broadcast_to(np.asarray(u, dtype=np.float64), g.shape)
    f = lib().orc_swiglu_oai
    return np.array([f(float(a), float(b), float(alpha), float(limit)) for a, b in zip(g.ravel(), u.ravel())]).reshape(g.shape)


def set_threads(n: int) -> None:
    """OpenMP threads for the oracle's parallel loops (n <= 0: all cores).
    Results are identical for any thread count."""
    lib().orc_set_threads(int(n))
