"""moe_permute_no_alloc: the permutation for callers that may not allocate
device memory (a framework plugin that owns no allocator, a serving loop that
must not call cudaMalloc).  It uses a static scratch array inside the library;
its output must equal moe_permute's (which uses a caller workspace) bit for
bit, on consecutive calls that reuse the shared array."""
import ctypes

import numpy as np
import pytest
import torch

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


def test_no_alloc_permute_rejects_oversized_requests(mx):
    L = mx.lib()
    fake = ctypes.c_void_p(256)   # never touched: the size check comes first
    assert L.moe_permute_no_alloc(fake, 8192, 1024, 32, fake, fake, fake, None) == mx.MX_ERR_WORKSPACE
