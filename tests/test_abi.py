"""Host-side tests of the C ABI (no GPU needed): the library builds, loads and
exports every entry point include/mxmoe.h declares, and argument validation
rejects bad calls before any device work is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxmoe.h")


@pytest.fixture(scope="module")
def L():
    from block_scaled_mx_gb300 import build as B
    from block_scaled_mx_gb300 import mxmoe as mx

    B.build()
    return mx.lib()


def _declared():
    txt = open(HEADER).read()
    return re.findall(r"^MX_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt, flags=re.M)


def test_header_declares_the_boundary():
    names = set(_declared())
    for n in ["mx_quantize_act", "moe_route_topk", "moe_permute", "moe_grouped_gemm_swiglu",
              "moe_grouped_gemm_down_combine", "moe_forward", "moe_prepare_weights", "moe_workspace_size",
              "moe_get_status", "mx_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    from block_scaled_mx_gb300 import mxmoe as mx

    for name in _declared():
        assert hasattr(L, name), name
        assert name in mx.SIGNATURES, f"binding lacks {name}"


def test_status_strings(L):
    for code in range(8):
        s = L.mx_status_string(code)
        assert s and s != b"unknown status"
    assert L.mx_status_string(99) == b"unknown status"


def test_sizes_are_host_only(L):
    assert L.moe_prepared_weight_bytes(9, 256, 128, 0, 1) > 9 * 256 * 256
    assert L.moe_prepared_weight_bytes(9, 256, 128, 1, 2) < L.moe_prepared_weight_bytes(9, 256, 128, 0, 2)
    assert L.moe_prepared_weight_bytes(9, 250, 128, 0, 1) == 0   # H % 128
    assert L.moe_permute_workspace_size(16, 8, 2) > 0
    assert L.moe_workspace_size(16, 256, 128, 8, 2, 0) > 16 * 3 * 256
    assert L.moe_workspace_size(16, 256, 100, 8, 2, 0) == 0      # I % 128
    assert L.moe_gemm_workspace_size(16, 256, 128, 8, 9) == 0   # k > E


def test_argument_validation_before_device_work(L):
    P = ctypes.c_void_p
    fake = P(256)   # never dereferenced: every call below fails validation first
    assert L.mx_quantize_act(None, 4, 64, fake, fake, None) == 1
    assert L.mx_quantize_act(fake, 4, 48, fake, fake, None) == 2
    assert L.mx_quantize_act(P(258), 4, 64, fake, fake, None) == 3
    assert L.mx_quantize_act(fake, 0, 64, None, None, None) == 0        # empty is a no-op
    assert L.moe_route_topk(fake, 4, 8, 9, fake, fake, None) == 1        # k > E
    assert L.moe_route_topk(fake, 4, 2000, 8, fake, fake, None) == 2     # E > 1024
    assert L.moe_route_topk(fake, 4, 64, 33, fake, fake, None) == 1      # k > 32
    assert L.moe_permute(fake, 4, 8, 2, fake, fake, fake, fake, 8, None) == 4   # workspace
    assert L.moe_prepare_weights(fake, fake, 9, 256, 100, 0, 1, fake, 1 << 30, None) == 2
    assert L.moe_prepare_weights(fake, fake, 9, 256, 128, 0, 1, P(272), 1 << 30, None) == 3
    assert L.moe_prepare_weights(fake, fake, 9, 256, 128, 0, 1, fake, 10, None) == 4
    assert L.moe_forward(fake, fake, fake, fake, 0, 4, 256, 128, 8, 2, fake, fake, 1, None) == 4
    assert L.moe_forward(fake, fake, fake, fake, 7, 4, 256, 128, 8, 2, fake, fake, 1 << 30, None) == 1
    assert L.moe_forward(fake, fake, fake, fake, 0, 4, 256, 128, 8, 2, fake, P(272), 1 << 30, None) == 3
    assert L.moe_grouped_gemm_swiglu(fake, fake, fake, fake, fake, 0, 4, 256, 128, 8, 2, fake, fake, fake, 1,
                                     None) == 4
    assert L.moe_grouped_gemm_down_combine(fake, fake, fake, fake, fake, fake, 0, 4, 200, 128, 8, 2, fake, fake,
                                           1 << 30, None) == 2


def test_product_does_not_import_oracle():
    pkg = os.path.join(ROOT, "block_scaled_mx_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
                assert "mx_oracle" not in txt, f


def test_binding_refuses_host_and_strided_tensors(L):
    """The binding hands the library plain device addresses: a host tensor or a
    strided view is refused before any call reaches the library."""
    import torch

    from block_scaled_mx_gb300 import mxmoe as mx

    host = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        mx.mx_quantize_act(host, None, None)
    meta = torch.empty(64, 4, dtype=torch.bfloat16, device="meta").t()
    assert not meta.is_contiguous()
    with pytest.raises(ValueError, match="contiguous"):
        mx._ptr(meta)
    assert mx._ptr(None) is None and mx._ptr(4096) == 4096


def test_loaded_library_is_built_from_these_sources(L):
    """The stamp compiled into the library equals the hash of the current
    sources, headers, flags and compiler (a stale or foreign build is rebuilt)."""
    from block_scaled_mx_gb300 import build as B

    assert L.mx_build_stamp().decode() == B.source_stamp() == B.built_stamp()


def test_forward_launch_count(L):
    """moe_forward's launch count is a host-side answer: three at decode sizes
    (prologue with the permutation, two grouped GEMMs), -1 for rejected shapes,
    0 for no tokens."""
    assert L.moe_forward_launches(32, 4096, 1536, 128, 8, 0) == 3
    assert L.moe_forward_launches(6, 2048, 512, 512, 8, 1) == 3
    assert L.moe_forward_launches(0, 256, 128, 8, 2, 0) == 0
    assert L.moe_forward_launches(16, 256, 100, 8, 2, 0) == -1
    assert L.moe_forward_launches(8192, 4096, 1536, 128, 8, 0) >= 3


def test_layer_options_are_checked_on_the_host(L):
    """mx_layer_opts: unknown values and a non-positive clamp limit are invalid
    arguments; MXFP4 activations with MXFP8 weights are unsupported; the
    dense shared-expert variant adds two launches."""
    from block_scaled_mx_gb300 import mxmoe as mx

    fake = ctypes.c_void_p(256)
    bad_act = mx.LayerOpts(7, 1.0, 7.0, 0, 0)
    bad_limit = mx.layer_opts("swiglu_oai", alpha=1.702, limit=0.0)
    bad_shared = mx.LayerOpts(0, 1.0, 7.0, 3, 0)
    for o in (bad_act, bad_limit, bad_shared):
        assert L.moe_forward_ex(fake, fake, fake, fake, 0, 4, 256, 128, 8, 2, fake, fake, 1 << 30, ctypes.addressof(o),
                                None) == mx.MX_ERR_INVALID_ARG
        assert L.moe_forward_launches_ex(32, 4096, 1536, 128, 8, 0, ctypes.addressof(o)) == -1
    # MXFP4 activations need MXFP4 weights (the packed-FP4 MMA takes E2M1 on both sides)
    fp4 = mx.layer_opts(act_fmt="e2m1")
    assert L.moe_forward_ex(fake, fake, fake, fake, 0, 4, 256, 128, 8, 2, fake, fake, 1 << 30,
                            ctypes.addressof(fp4), None) == mx.MX_ERR_UNSUPPORTED
    assert L.moe_grouped_gemm_swiglu_ex(fake, fake, fake, fake, fake, 0, 4, 256, 128, 8, 2, fake, fake, fake,
                                        1 << 30, ctypes.addressof(fp4), None) == mx.MX_ERR_UNSUPPORTED
    assert L.moe_grouped_gemm_down_combine_ex(fake, fake, fake, fake, fake, fake, 0, 4, 256, 128, 8, 2, fake, fake,
                                              1 << 30, ctypes.addressof(fp4), None) == mx.MX_ERR_UNSUPPORTED
    assert L.mx_quantize_act_ex(fake, 4, 256, 7, fake, fake, None) == mx.MX_ERR_INVALID_ARG
    dense = mx.layer_opts(shared="dense")
    assert L.moe_forward_launches_ex(32, 4096, 1536, 128, 8, 0, ctypes.addressof(dense)) == 5
    assert L.moe_forward_launches_ex(32, 4096, 1536, 128, 8, 0, None) == 3
    assert mx.moe_forward_launches_ex(32, 4096, 1536, 128, 8, "e4m3", mx.layer_opts("swiglu_oai")) == 3


def test_gemm_timing_hook_without_launches(L):
    """The timing hook makes no CUDA call until a GEMM launch is recorded:
    enabling, reading (nothing recorded) and disabling work without a GPU."""
    from block_scaled_mx_gb300 import mxmoe as mx

    mx.mx_debug_time_gemms(True)
    assert mx.mx_debug_gemm_times() == ([], [])
    mx.mx_debug_time_gemms(False)
    assert L.mx_debug_gemm_times(None, None, 0) == 0
