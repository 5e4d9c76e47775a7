"""moe_permute_no_alloc: the permutation for callers that may not allocate
device memory (a framework plugin that owns no allocator, a serving loop that
must not call cudaMalloc).  It uses a static scratch array inside the library;
its output must equal moe_permute's (which uses a caller workspace) bit for
bit, on consecutive calls that reuse the shared array."""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g

    g.build()
    torch.cuda.set_device(0)
    from block_scaled_mx_gb300 import mxmoe

    return mxmoe


def _ids(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g)
    logits[:, seed % E] += 2.0   # one popular expert
    return torch.topk(logits, k, dim=1).indices.to(torch.int32).cuda()


def _run(mx, fn, ids, E):
    T, k = ids.shape
    counts = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 2,), -1, dtype=torch.int32, device="cuda")
    ss = torch.full((T * (k + 1),), -1, dtype=torch.int32, device="cuda")
    fn(ids, counts, offsets, ss)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), offsets.cpu().numpy(), ss.cpu().numpy()


def test_no_alloc_permute_matches_workspace_permute(mx):
    cases = [(300, 128, 8, 1), (8192, 512, 8, 2), (6, 512, 8, 3), (1000, 64, 4, 4)]
    for T, E, k, seed in cases:   # consecutive calls share and reuse the static scratch
        ids = _ids(T, E, k, seed)
        ws = mx.alloc_workspace(mx.moe_permute_workspace_size(T, E, k))
        ref = _run(mx, lambda i, c, o, s: mx.moe_permute(i, E, c, o, s, ws), ids, E)
        for _ in range(2):
            got = _run(mx, lambda i, c, o, s: mx.moe_permute_no_alloc(i, E, c, o, s), ids, E)
            for a, b in zip(got, ref):
                assert np.array_equal(a, b), (T, E, k)


def _tied_ids(T, E, k, seed):
    """Top-k of small-integer logits: many equal logits per token, so the ids
    come from the lowest-index tie-break and many tokens share experts."""
    g = torch.Generator().manual_seed(seed)
    logits = torch.randint(-1, 2, (T, E), generator=g).float()
    ids, _ = oracle.route_topk(logits.numpy(), k)
    return torch.from_numpy(ids).cuda()


def _same_as_workspace_form(mx, ids, E):
    T, k = ids.shape
    ws = mx.alloc_workspace(mx.moe_permute_workspace_size(T, E, k))
    ref = _run(mx, lambda i, c, o, s: mx.moe_permute(i, E, c, o, s, ws), ids, E)
    got = _run(mx, lambda i, c, o, s: mx.moe_permute_no_alloc(i, E, c, o, s), ids, E)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b), (T, E, k)


def test_no_alloc_permute_shape_changes_between_calls(mx):
    """The shared array keeps the previous call's chunk tables and ranks: a
    one-chunk call straight after a many-chunk call on another expert count,
    and the reverse, must not see them."""
    for T, E, k, seed in [(5000, 256, 6, 11), (40, 32, 4, 12), (7000, 96, 8, 13), (3, 512, 8, 14),
                          (257, 8, 2, 15), (256, 64, 3, 16)]:
        _same_as_workspace_form(mx, _ids(T, E, k, seed), E)


def test_no_alloc_permute_ties(mx):
    """Routing full of equal logits: many tokens per expert and ids that come
    from the tie-break, one chunk and several chunks."""
    for T, E, k, seed in [(200, 16, 4, 21), (3000, 64, 8, 22), (9, 8, 8, 23)]:
        _same_as_workspace_form(mx, _tied_ids(T, E, k, seed), E)


def test_no_alloc_permute_rejects_oversized_requests(mx):
    L = mx.lib()
    fake = ctypes.c_void_p(256)   # never touched: the size check comes first
    assert L.moe_permute_no_alloc(fake, 8192, 1024, 32, fake, fake, fake, None) == mx.MX_ERR_WORKSPACE
