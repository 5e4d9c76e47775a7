"""ctypes binding of libmxmoe.so (see include/mxmoe.h for every call's contract).

Argument marshalling only: tensors become device pointers, the stream defaults
to torch's current stream, a non-zero status raises ``MxError``.  All compute
runs in the library's CUDA kernels; there is no fallback: if the library is
missing or no GPU is present the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# MXMOE_LIB selects another build of the same library (e.g. a tuning variant)
LIB_PATH = os.environ.get("MXMOE_LIB") or os.path.join(_HERE, "libmxmoe.so")

MX_OK = 0
MX_ERR_INVALID_ARG = 1
MX_ERR_UNSUPPORTED = 2
MX_ERR_ALIGNMENT = 3
MX_ERR_WORKSPACE = 4
MX_ERR_CUDA = 5
MX_ERR_TIMEOUT = 6
MX_ERR_DEVICE_ARG = 7
MX_E4M3 = 0
MX_E2M1 = 1
FORMATS = {"e4m3": MX_E4M3, "e2m1": MX_E2M1}
MX_ACT_SWIGLU = 0
MX_ACT_SWIGLU_OAI = 1
MX_SHARED_FOLDED = 0
MX_SHARED_DENSE = 1


class LayerOpts(ctypes.Structure):
    """mx_layer_opts of include/mxmoe.h (field order and types as declared)."""
    _fields_ = [("activation", ctypes.c_int), ("alpha", ctypes.c_float), ("limit", ctypes.c_float),
                ("shared_expert", ctypes.c_int), ("act_fmt", ctypes.c_int)]


def layer_opts(activation="swiglu", alpha=1.0, limit=7.0, shared="folded", act_fmt="e4m3") -> LayerOpts:
    """Options from names: activation "swiglu" | "swiglu_oai", shared "folded" | "dense"."""
    return LayerOpts({"swiglu": MX_ACT_SWIGLU, "swiglu_oai": MX_ACT_SWIGLU_OAI}[activation], float(alpha),
                     float(limit), {"folded": MX_SHARED_FOLDED, "dense": MX_SHARED_DENSE}[shared],
                     FORMATS[act_fmt] if isinstance(act_fmt, str) else int(act_fmt))

# every entry point of the C ABI: name -> (restype, argtypes)
_P, _I, _I64, _SZ, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint64
SIGNATURES = {
    "mx_status_string": (ctypes.c_char_p, [_I]),
    "mx_quantize_act": (_I, [_P, _I, _I, _P, _P, _P]),
    "mx_quantize_act_ex": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "mx_quantize_weights": (_I, [_P, _I64, _I, _I, _P, _P, _P]),
    "moe_route_topk": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_route_gemm_topk": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_workspace_size": (_SZ, [_I, _I, _I]),
    "moe_permute": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_no_alloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _P]),
    "moe_prepared_weight_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_prepare_weights": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "moe_gemm_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_grouped_gemm_swiglu": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "moe_grouped_gemm_down_combine": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_grouped_gemm_down_combine_ex": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P]),
    "moe_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_forward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_forward_ex": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P]),
    "moe_grouped_gemm_swiglu_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P, _P]),
    "moe_forward_launches_ex": (_I, [_I, _I, _I, _I, _I, _I, _P]),
    "moe_forward_launches": (_I, [_I, _I, _I, _I, _I, _I]),
    "moe_get_status": (_I, [_P, _P, _P]),
    "mx_debug_set_wait_limit_ns": (None, [_U64]),
    "mx_debug_time_gemms": (None, [_I]),
    "mx_debug_gemm_times": (_I, [_P, _P, _I]),
    "mx_build_stamp": (ctypes.c_char_p, []),
}

_lib = None


class MxError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


def lib(path: Optional[str] = None):
    """Load libmxmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None or path:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libmxmoe.so not built ({p}); run __graft_entry__.build()")
        L = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        if path:
            return L
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().mx_status_string(status).decode()
    except Exception:
        return f"status {status}"


def _ptr(t) -> Optional[int]:
    """A tensor's device address.  The library reads every buffer as dense
    row-major device memory, so a strided view or a host tensor is refused
    here rather than read wrongly.  An int is taken as a raw device pointer."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got shape {tuple(t.shape)} strides {t.stride()}")
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, what: str):
    if st != MX_OK:
        raise MxError(st, what)


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


# ------------------------------------------------------------------ step calls
def mx_quantize_act(x, codes, scales, stream=None, fmt=None):
    """x bf16 [T, H] -> MX codes and E8M0 scales; fmt None/"e4m3" (codes [T, H])
    or "e2m1" (MXFP4, codes [T, H/2])."""
    T, H = x.shape
    if fmt is None:
        _check(lib().mx_quantize_act(_ptr(x), T, H, _ptr(codes), _ptr(scales), _stream(stream)), "mx_quantize_act")
    else:
        _check(lib().mx_quantize_act_ex(_ptr(x), T, H, _fmt(fmt), _ptr(codes), _ptr(scales), _stream(stream)),
               "mx_quantize_act_ex")


def mx_quantize_weights(w, fmt, codes, scales, stream=None):
    rows, K = w.shape
    _check(lib().mx_quantize_weights(_ptr(w), rows, K, _fmt(fmt), _ptr(codes), _ptr(scales), _stream(stream)),
           "mx_quantize_weights")


def moe_route_topk(logits, k, topk_ids, topk_w, stream=None):
    T, E = logits.shape
    _check(lib().moe_route_topk(_ptr(logits), T, E, k, _ptr(topk_ids), _ptr(topk_w), _stream(stream)),
           "moe_route_topk")


def moe_route_gemm_topk(x, w_router, k, ws, bias=None, logits=None, topk_ids=None, topk_w=None, stream=None):
    """Router GEMM (bf16 x [T, H] . w_router [E, H]^T, fp32) with top-k in its
    epilogue; logits, ids and weights are written where tensors are given."""
    T, H = x.shape
    E = w_router.shape[0]
    _check(lib().moe_route_gemm_topk(_ptr(x), _ptr(w_router), _ptr(bias), T, H, E, k, _ptr(logits), _ptr(topk_ids),
                                     _ptr(topk_w), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_route_gemm_topk")


def moe_permute_workspace_size(T, E, k) -> int:
    return lib().moe_permute_workspace_size(T, E, k)


def moe_permute(topk_ids, E, counts, offsets, sorted_slot, ws, stream=None):
    T, k = topk_ids.shape
    _check(lib().moe_permute(_ptr(topk_ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(sorted_slot), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream)), "moe_permute")


def moe_permute_no_alloc(topk_ids, E, counts, offsets, sorted_slot, stream=None):
    """moe_permute with the library's own static scratch (for callers that may not allocate)."""
    T, k = topk_ids.shape
    _check(lib().moe_permute_no_alloc(_ptr(topk_ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(sorted_slot),
                                      _stream(stream)), "moe_permute_no_alloc")


def moe_prepared_weight_bytes(E1, H, I, fmt, which) -> int:
    return lib().moe_prepared_weight_bytes(E1, H, I, _fmt(fmt), which)


def moe_prepare_weights(codes, scales, E1, H, I, fmt, which, dst, stream=None):
    _check(lib().moe_prepare_weights(_ptr(codes), _ptr(scales), E1, H, I, _fmt(fmt), which, _ptr(dst),
                                     dst.numel() * dst.element_size(), _stream(stream)), "moe_prepare_weights")


def moe_gemm_workspace_size(T, H, I, E, k) -> int:
    return lib().moe_gemm_workspace_size(T, H, I, E, k)


def moe_grouped_gemm_swiglu(act_codes, act_scales, offsets, sorted_slot, w1_prep, fmt, T, H, I, E, k, h_codes,
                            h_scales, ws, stream=None):
    _check(lib().moe_grouped_gemm_swiglu(_ptr(act_codes), _ptr(act_scales), _ptr(offsets), _ptr(sorted_slot),
                                         _ptr(w1_prep), _fmt(fmt), T, H, I, E, k, _ptr(h_codes), _ptr(h_scales),
                                         _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_grouped_gemm_swiglu")


def _opts_ptr(opts):
    return None if opts is None else ctypes.addressof(opts)


def moe_grouped_gemm_swiglu_ex(act_codes, act_scales, offsets, sorted_slot, w1_prep, fmt, T, H, I, E, k, h_codes,
                               h_scales, ws, opts=None, stream=None):
    _check(lib().moe_grouped_gemm_swiglu_ex(_ptr(act_codes), _ptr(act_scales), _ptr(offsets), _ptr(sorted_slot),
                                            _ptr(w1_prep), _fmt(fmt), T, H, I, E, k, _ptr(h_codes), _ptr(h_scales),
                                            _ptr(ws), ws.numel() * ws.element_size(), _opts_ptr(opts),
                                            _stream(stream)), "moe_grouped_gemm_swiglu_ex")


def moe_grouped_gemm_down_combine(h_codes, h_scales, offsets, sorted_slot, topk_w, w2_prep, fmt, T, H, I, E, k,
                                  out, ws, stream=None, opts=None):
    if opts is None:
        _check(lib().moe_grouped_gemm_down_combine(_ptr(h_codes), _ptr(h_scales), _ptr(offsets), _ptr(sorted_slot),
                                                   _ptr(topk_w), _ptr(w2_prep), _fmt(fmt), T, H, I, E, k, _ptr(out),
                                                   _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
               "moe_grouped_gemm_down_combine")
    else:
        _check(lib().moe_grouped_gemm_down_combine_ex(_ptr(h_codes), _ptr(h_scales), _ptr(offsets),
                                                      _ptr(sorted_slot), _ptr(topk_w), _ptr(w2_prep), _fmt(fmt), T,
                                                      H, I, E, k, _ptr(out), _ptr(ws),
                                                      ws.numel() * ws.element_size(), _opts_ptr(opts),
                                                      _stream(stream)),
               "moe_grouped_gemm_down_combine_ex")


def moe_workspace_size(T, H, I, E, k, fmt) -> int:
    return lib().moe_workspace_size(T, H, I, E, k, _fmt(fmt))


def moe_forward(x, logits, w1_prep, w2_prep, fmt, I, k, out, ws, stream=None):
    T, H = x.shape
    E = logits.shape[1]
    _check(lib().moe_forward(_ptr(x), _ptr(logits), _ptr(w1_prep), _ptr(w2_prep), _fmt(fmt), T, H, I, E, k,
                             _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_forward")


def moe_forward_launches(T, H, I, E, k, fmt) -> int:
    """Kernel launches moe_forward enqueues for this shape (host only)."""
    return lib().moe_forward_launches(T, H, I, E, k, _fmt(fmt))


def moe_forward_ex(x, logits, w1_prep, w2_prep, fmt, I, k, out, ws, opts=None, stream=None):
    T, H = x.shape
    E = logits.shape[1]
    _check(lib().moe_forward_ex(_ptr(x), _ptr(logits), _ptr(w1_prep), _ptr(w2_prep), _fmt(fmt), T, H, I, E, k,
                                _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _opts_ptr(opts),
                                _stream(stream)), "moe_forward_ex")


def moe_forward_launches_ex(T, H, I, E, k, fmt, opts=None) -> int:
    """Kernel launches moe_forward_ex enqueues for this shape and these options (host only)."""
    return lib().moe_forward_launches_ex(T, H, I, E, k, _fmt(fmt), _opts_ptr(opts))


def moe_get_status(ws, stream=None) -> int:
    v = ctypes.c_int(0)
    _check(lib().moe_get_status(_ptr(ws), _stream(stream), ctypes.addressof(v)), "moe_get_status")
    return v.value


def mx_debug_set_wait_limit_ns(ns: int):
    lib().mx_debug_set_wait_limit_ns(int(ns))


def mx_debug_time_gemms(enable: bool):
    """Start (or stop) bracketing each grouped-GEMM launch with CUDA events."""
    lib().mx_debug_time_gemms(1 if enable else 0)


def mx_debug_gemm_times(max_n: int = 4096):
    """Device times (ms) and epilogues (0 gate/up, 1 down) of the grouped-GEMM
    launches recorded since timing was enabled or last read; clears them."""
    ms = (ctypes.c_float * max_n)()
    epi = (ctypes.c_int * max_n)()
    n = lib().mx_debug_gemm_times(ctypes.cast(ms, _P), ctypes.cast(epi, _P), max_n)
    if n < 0:
        raise MxError(MX_ERR_CUDA, "mx_debug_gemm_times")
    n = min(n, max_n)
    return [float(ms[i]) for i in range(n)], [int(epi[i]) for i in range(n)]


def mx_build_stamp() -> str:
    """Hash of the sources and flags the loaded library was compiled from."""
    return lib().mx_build_stamp().decode()


# ------------------------------------------------------------------ buffers (caller-owned memory)
def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled, 256-byte aligned workspace (the library requires zero on first use)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class MoELayer:
    """One MoE expert layer with prepared MX weights resident on the GPU.

    ``w1_codes/w1_scales``: canonical [E+1, 2I, H(/2)] / [E+1, 2I, H/32];
    ``w2_codes/w2_scales``: [E+1, H, I(/2)] / [E+1, H, I/32]; shared expert last."""

    def __init__(self, w1_codes, w1_scales, w2_codes, w2_scales, fmt, H, I, E, k, stream=None):
        self.fmt, self.H, self.I, self.E, self.k = _fmt(fmt), H, I, E, k
        dev = w1_codes.device
        self.w1 = torch.empty(moe_prepared_weight_bytes(E + 1, H, I, fmt, 1), dtype=torch.uint8, device=dev)
        self.w2 = torch.empty(moe_prepared_weight_bytes(E + 1, H, I, fmt, 2), dtype=torch.uint8, device=dev)
        moe_prepare_weights(w1_codes, w1_scales, E + 1, H, I, fmt, 1, self.w1, stream)
        moe_prepare_weights(w2_codes, w2_scales, E + 1, H, I, fmt, 2, self.w2, stream)
        self._ws = None

    def workspace(self, T: int, device="cuda") -> torch.Tensor:
        need = moe_workspace_size(T, self.H, self.I, self.E, self.k, self.fmt)
        if self._ws is None or self._ws.numel() < need:
            self._ws = alloc_workspace(need, device)
        return self._ws

    def forward(self, x, logits, out=None, stream=None, opts: Optional[LayerOpts] = None) -> torch.Tensor:
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.float32, device=x.device)
        if opts is None:
            moe_forward(x, logits, self.w1, self.w2, self.fmt, self.I, self.k, out, self.workspace(T, x.device),
                        stream)
        else:
            moe_forward_ex(x, logits, self.w1, self.w2, self.fmt, self.I, self.k, out, self.workspace(T, x.device),
                           opts, stream)
        return out
