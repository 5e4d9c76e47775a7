"""Device-side failure reporting without faulting the GPU: every wait inside the
grouped GEMM kernel is bounded; shortening the bound makes the waits run out,
which must surface as MX_ERR_TIMEOUT in the workspace status word, and the next
call with the normal bound must run correctly on the same context."""
import numpy as np
import pytest
import torch

from block_scaled_mx_gb300 import mxmoe as mx
from block_scaled_mx_gb300 import workload as W

from layer_inputs import OUT_MAX_ABS_OVER_RMS, OUT_REL_L2, build_layer, oracle_forward, out_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g

    g.build()
    torch.cuda.set_device(0)


def test_wait_timeout_is_reported_and_context_survives():
    wl = W.WORKLOADS["tiny"]
    L = build_layer(wl)
    ref = oracle_forward(L)["out"]
    ws = L.layer.workspace(wl.T)
    try:
        mx.mx_debug_set_wait_limit_ns(0)
        L.layer.forward(L.x, L.logits)
        st = mx.moe_get_status(ws)
    finally:
        mx.mx_debug_set_wait_limit_ns(2_000_000_000)
    assert st == mx.MX_ERR_TIMEOUT
    out = L.layer.forward(L.x, L.logits)
    assert mx.moe_get_status(ws) == 0
    rel, mabs = out_errors(out.double().cpu().numpy(), ref)
    assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS


def test_out_of_range_expert_id_is_reported():
    T, E, k = 40, 16, 2
    ids = torch.randint(0, E, (T, k), dtype=torch.int32)
    ids[:, 1] = (ids[:, 0] + 1) % E
    ids[7, 1] = E + 3           # invalid id: skipped and flagged
    ids = ids.cuda()
    counts = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 2, dtype=torch.int32, device="cuda")
    ss = torch.empty(T * (k + 1), dtype=torch.int32, device="cuda")
    ws = mx.alloc_workspace(mx.moe_permute_workspace_size(T, E, k))
    mx.moe_permute(ids, E, counts, offsets, ss, ws)
    assert mx.moe_get_status(ws) == mx.MX_ERR_DEVICE_ARG
    assert int(counts[:E].sum()) == T * k - 1
