"""GPU parity of the router GEMM with top-k in its epilogue
(moe_route_gemm_topk) against the oracle.

logits: fp32 tensor-core accumulation of exact bf16 products against the
oracle's fp64 sums, within a bound from the fp32 rounding of a sum of H terms.
ids: bit-exact against the oracle's biased top-k run on the GPU's own fp32
logits (both sides take the selection decision on the same fp32 values).
weights: fp32 softmax against fp64, rtol 2e-6."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_mx_gb300 import mxmoe as mx

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g

    g.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _inputs(T, H, E, seed, bias_scale):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    bias = (torch.randn(E, generator=g) * bias_scale).float() if bias_scale else None
    return x, w, bias


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


CASES = [(16, 256, 8, 2), (32, 4096, 128, 8), (6, 2048, 512, 8), (1000, 512, 128, 8), (70, 192, 100, 16),
         (300, 128, 300, 4)]


@pytest.mark.parametrize("T,H,E,k", CASES)
@pytest.mark.parametrize("bias_scale", [0.0, 0.5])
def test_router_parity(T, H, E, k, bias_scale):
    x, w, bias = _inputs(T, H, E, T + H + E, bias_scale)
    ws = mx.alloc_workspace(256)
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    tw = torch.empty(T, k, dtype=torch.float32, device="cuda")
    mx.moe_route_gemm_topk(x.cuda(), w.cuda(), k, ws, bias=None if bias is None else bias.cuda(), logits=logits,
                           topk_ids=ids, topk_w=tw)
    assert mx.moe_get_status(ws) == 0
    got = logits.cpu().numpy()
    ref = oracle.router_logits(_bits(x), _bits(w))
    # fp32 accumulation of H exact products: error below H * 2^-24 * sum |x w|
    absum = np.abs(x.double().numpy()) @ np.abs(w.double().numpy()).T
    assert np.all(np.abs(got - ref) <= H * 2.0 ** -24 * absum + 1e-30)
    rid, rw = oracle.route_topk_biased(got, None if bias is None else bias.numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(tw.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)
    if bias is None:
        # the same selection as the stand-alone top-k on these logits
        ids2 = torch.empty_like(ids)
        tw2 = torch.empty_like(tw)
        mx.moe_route_topk(logits, k, ids2, tw2)
        assert torch.equal(ids2, ids)


@pytest.mark.parametrize("T,H,E,k", [(40, 128, 64, 8), (130, 256, 100, 16), (20, 192, 512, 8), (9, 64, 8, 8)])
def test_router_logits_only_and_ties(T, H, E, k):
    """Logits without selection; and exactly tied scores (integer inputs make
    the logits exact) resolve to the lowest expert index."""
    g = torch.Generator().manual_seed(T + E)
    x = torch.randint(-1, 2, (T, H), generator=g).to(torch.bfloat16)
    w = torch.randint(-1, 2, (E, H), generator=g).to(torch.bfloat16)
    w[E - 1] = w[1]   # experts 1 and E - 1 tie for every token
    ws = mx.alloc_workspace(256)
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    mx.moe_route_gemm_topk(x.cuda(), w.cuda(), k, ws, logits=logits)
    ref = oracle.router_logits(_bits(x), _bits(w))
    assert np.array_equal(logits.cpu().numpy().astype(np.float64), ref)   # integer sums are exact
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    tw = torch.empty(T, k, dtype=torch.float32, device="cuda")
    mx.moe_route_gemm_topk(x.cuda(), w.cuda(), k, ws, topk_ids=ids, topk_w=tw)
    rid, rw = oracle.route_topk_biased(ref.astype(np.float32), None, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(tw.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)
    assert mx.moe_get_status(ws) == 0


@pytest.mark.parametrize("T,H,E,k", [(32, 4096, 128, 8), (6, 2048, 512, 8), (64, 320, 40, 5), (1, 64, 8, 1),
                                     (128, 4096, 128, 8), (97, 192, 300, 16)])
def test_router_small_batch_without_caller_logits(T, H, E, k):
    """Up to 128 tokens the logits may live in a larger workspace instead of a
    caller buffer (the small-batch kernel); the selection matches the run that
    returns its logits, and both match the oracle's selection on those logits."""
    x, w, bias = _inputs(T, H, E, 7 * T + E, 0.5)
    xd, wd, bd = x.cuda(), w.cuda(), bias.cuda()
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    tw = torch.empty(T, k, dtype=torch.float32, device="cuda")
    ws = mx.alloc_workspace(256)
    mx.moe_route_gemm_topk(xd, wd, k, ws, bias=bd, logits=logits, topk_ids=ids, topk_w=tw)
    big = mx.alloc_workspace(256 + 4 * T * E)
    ids2 = torch.empty_like(ids)
    tw2 = torch.empty_like(tw)
    for _ in range(2):  # the block counter is ready again after a call
        mx.moe_route_gemm_topk(xd, wd, k, big, bias=bd, topk_ids=ids2, topk_w=tw2)
        assert torch.equal(ids2, ids)
        assert torch.equal(tw2, tw)
    assert mx.moe_get_status(ws) == 0 and mx.moe_get_status(big) == 0
    got = logits.cpu().numpy()
    ref = oracle.router_logits(_bits(x), _bits(w))
    absum = np.abs(x.double().numpy()) @ np.abs(w.double().numpy()).T
    assert np.all(np.abs(got - ref) <= H * 2.0 ** -24 * absum + 1e-30)
    rid, rw = oracle.route_topk_biased(got, bias.numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(tw.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)
