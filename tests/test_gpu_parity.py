"""GPU parity: every C-ABI call against the CPU oracle on the same seeded inputs.

Bit-exact: activation codes/scales, weight codes/scales (both formats), top-k
ids, counts, offsets, sorted slots.  Tolerances: top-k weights (fp32 softmax
vs fp64), h codes (fp32 tensor-core accumulation can move a value across a
rounding boundary: mismatch fraction reported and bounded), and the layer
output: relative L2 <= 5e-3 and max-abs <= 3% of the output RMS."""
import numpy as np
import pytest
import torch

import oracle
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
    yield
    torch.cuda.synchronize()


def _bf16(T, H, seed, scale_rows=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g)
    if scale_rows:
        x = x * torch.exp(torch.randn(T, 1, generator=g) * 3)
    return x.to(torch.bfloat16)


# ------------------------------------------------------------------ quantisers
@pytest.mark.parametrize("T,H", [(1, 32), (16, 256), (37, 4096), (6, 2048), (8192, 4096)])
def test_quantize_act_bitexact(T, H):
    x = _bf16(T, H, T * 7 + H)
    if T > 2:
        x[0, :32] = 0.0
        x[1, 3] = -1e-30          # negative that rounds to -0
        x[2, :32] = 1.0e-39       # all-subnormal bf16 block
        x[2, 40] = 3.0e38         # near the bf16 maximum
    xd = x.cuda()
    codes = torch.empty(T, H, dtype=torch.uint8, device="cuda")
    scales = torch.empty(T, H // 32, dtype=torch.uint8, device="cuda")
    mx.mx_quantize_act(xd, codes, scales)
    rc, rs = oracle.quantize_bf16(W.bf16_bits(x))
    assert np.array_equal(scales.cpu().numpy(), rs)
    got = codes.cpu().numpy()
    assert np.array_equal(got, rc), f"{np.count_nonzero(got != rc)} code mismatches"


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("rows,K,std", [(3, 32, 1.0), (256, 4096, 0.02), (129, 1536, 0.02), (64, 128, 1e-20)])
def test_quantize_weights_bitexact(fmt, rows, K, std):
    g = torch.Generator().manual_seed(rows + K)
    w = torch.randn(rows, K, generator=g) * std
    w[0, :32] = 0.0
    w[0, 5] = -1e-12      # a negative that rounds to -0 inside a zero-amax-dominated block
    if K > 32:
        w[0, 40] = -1e-12
    if rows > 2:
        w[1, :32] *= 1e-30   # tiny block
        w[2, 5] = 7.9        # E2M1 saturation region
    f = mx.FORMATS[fmt]
    cdiv = 1 if f == mx.MX_E4M3 else 2
    codes = torch.empty(rows, K // cdiv, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, K // 32, dtype=torch.uint8, device="cuda")
    mx.mx_quantize_weights(w.cuda(), f, codes, scales)
    rc, rs = oracle.quantize_f32(w.numpy(), f)
    assert np.array_equal(scales.cpu().numpy(), rs)
    got = codes.cpu().numpy()
    assert np.array_equal(got, rc), f"{np.count_nonzero(got != rc)} code mismatches"


# ------------------------------------------------------------------ router, permutation
@pytest.mark.parametrize("T,E,k,ties", [(16, 8, 2, False), (32, 128, 8, False), (6, 512, 8, False),
                                        (100, 64, 4, True), (3, 8, 8, True), (8192, 128, 8, False),
                                        (5, 1000, 32, False)])
def test_topk(T, E, k, ties):
    g = torch.Generator().manual_seed(T + E)
    if ties:
        logits = torch.randint(-2, 3, (T, E), generator=g).float()
    else:
        logits = torch.randn(T, E, generator=g)
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    mx.moe_route_topk(logits.cuda(), k, ids, w)
    rid, rw = oracle.route_topk(logits.numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (16, 8, 2), (32, 128, 8), (6, 512, 8), (300, 16, 4),
                                   (8192, 128, 8), (513, 1024, 3)])
def test_permute_bitexact(T, E, k):
    g = torch.Generator().manual_seed(T * 3 + E)
    logits = torch.randn(T, E, generator=g)
    if T >= 300:
        logits[:, 0] += 3.0   # a skewed expert
    rid, _ = oracle.route_topk(logits.numpy(), k)
    ids = torch.from_numpy(rid).cuda()
    counts = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 2, dtype=torch.int32, device="cuda")
    ss = torch.empty(T * (k + 1), dtype=torch.int32, device="cuda")
    ws = mx.alloc_workspace(mx.moe_permute_workspace_size(T, E, k))
    for _ in range(2):   # second call checks the workspace is left ready
        ss.fill_(-1)
        mx.moe_permute(ids, E, counts, offsets, ss, ws)
        rc, ro, rs = oracle.permute(rid, E)
        assert np.array_equal(counts.cpu().numpy(), rc)
        assert np.array_equal(offsets.cpu().numpy(), ro)
        assert np.array_equal(ss.cpu().numpy(), rs)
    assert mx.moe_get_status(ws) == 0


# ------------------------------------------------------------------ layer
def _steps(L, opts=None):
    wl = L.wl
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    d = "cuda"
    r = {}
    r["act_c"] = torch.empty(T, H, dtype=torch.uint8, device=d)
    r["act_s"] = torch.empty(T, H // 32, dtype=torch.uint8, device=d)
    mx.mx_quantize_act(L.x, r["act_c"], r["act_s"])
    r["ids"] = torch.empty(T, k, dtype=torch.int32, device=d)
    r["w"] = torch.empty(T, k, dtype=torch.float32, device=d)
    mx.moe_route_topk(L.logits, k, r["ids"], r["w"])
    r["counts"] = torch.empty(E + 1, dtype=torch.int32, device=d)
    r["offsets"] = torch.empty(E + 2, dtype=torch.int32, device=d)
    r["ss"] = torch.empty(T * (k + 1), dtype=torch.int32, device=d)
    pws = mx.alloc_workspace(mx.moe_permute_workspace_size(T, E, k))
    mx.moe_permute(r["ids"], E, r["counts"], r["offsets"], r["ss"], pws)
    gws = mx.alloc_workspace(mx.moe_gemm_workspace_size(T, H, I, E, k))
    r["h_c"] = torch.empty(T * (k + 1), I, dtype=torch.uint8, device=d)
    r["h_s"] = torch.empty(T * (k + 1), I // 32, dtype=torch.uint8, device=d)
    if opts is None:
        mx.moe_grouped_gemm_swiglu(r["act_c"], r["act_s"], r["offsets"], r["ss"], L.layer.w1, L.fmt, T, H, I, E, k,
                                   r["h_c"], r["h_s"], gws)
    else:
        mx.moe_grouped_gemm_swiglu_ex(r["act_c"], r["act_s"], r["offsets"], r["ss"], L.layer.w1, L.fmt, T, H, I, E,
                                      k, r["h_c"], r["h_s"], gws, opts)
    r["out"] = torch.zeros(T, H, dtype=torch.float32, device=d)
    mx.moe_grouped_gemm_down_combine(r["h_c"], r["h_s"], r["offsets"], r["ss"], r["w"], L.layer.w2, L.fmt, T, H,
                                     I, E, k, r["out"], gws)
    r["status"] = (mx.moe_get_status(pws), mx.moe_get_status(gws))
    return r


def _signed_code_index(c):
    """E4M3 code -> signed position on the value grid (+0 and -0 both 0):
    magnitudes grow with the low seven bits, so neighbours differ by one."""
    c = c.astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def _e4m3_quantum(v, scale_codes):
    """Spacing of the E4M3 grid at |v| under the block scale 2^(code - 127):
    2^(e - 3) in the binade 2^e of |v| / scale, 2^-9 below 2^-6."""
    S = np.exp2(scale_codes.astype(np.float64) - 127)
    a = np.maximum(np.abs(v) / S, 2.0 ** -6)
    _, ex = np.frexp(a)
    return S * np.exp2(ex - 1 - 3)


def _check_h(r, ref, I):
    """h codes against the oracle (GPU rows are slot positions, oracle rows are
    slot ids).  fp32 tensor-core accumulation can move a value across an E4M3
    rounding boundary (one code step), or move a block's amax across a power of
    two (the block's scale moves by one and its codes re-round): every mismatch
    must be one of those.  Returns (mismatch fraction, relative L2 of the
    decoded h)."""
    ss = r["ss"].cpu().numpy()
    gc = r["h_c"].cpu().numpy()
    gs = r["h_s"].cpu().numpy()
    rc = ref["h_codes"][ss]
    rs = ref["h_scales"][ss]
    gv = oracle.decode_matrix(gc, gs, oracle.E4M3)
    rv = oracle.decode_matrix(rc, rs, oracle.E4M3)
    gs_e = np.repeat(gs, 32, axis=1)
    rs_e = np.repeat(rs, 32, axis=1)
    same_scale = gs_e == rs_e
    assert np.all(np.abs(gs.astype(np.int64) - rs.astype(np.int64)) <= 1), "a block scale moved by more than one"
    step = np.abs(_signed_code_index(gc) - _signed_code_index(rc))
    assert np.all(step[same_scale] <= 1), "a code moved by more than one step under the same scale"
    coarse = np.maximum(gs_e, rs_e)
    moved = ~same_scale
    tol = _e4m3_quantum(np.maximum(np.abs(gv), np.abs(rv))[moved], coarse[moved])
    assert np.all(np.abs(gv - rv)[moved] <= tol), "a re-scaled value moved by more than one step of the coarser scale"
    frac = np.count_nonzero(gc != rc) / gc.size
    rel = np.linalg.norm(gv - rv) / np.linalg.norm(rv)
    return frac, rel


LAYER_CASES = {
    "tiny": W.WORKLOADS["tiny"],
    "decode_mxfp8": W.WORKLOADS["decode_mxfp8"],
    "decode_mxfp4": W.WORKLOADS["decode_mxfp4"],
    "specverify_mxfp4": W.WORKLOADS["specverify_mxfp4"],
    # ragged shapes: two permutation chunks, H = 3*128 (half last down tile)
    "ragged_e4m3": W.custom("ragged_e4m3", T=300, H=384, I=256, E=16, k=4, fmt="e4m3"),
    "ragged_e2m1": W.custom("ragged_e2m1", T=77, H=640, I=384, E=12, k=3, fmt="e2m1"),
    # wide (prefill) schedule with several ragged token tiles per expert
    "wide_e4m3": W.custom("wide_e4m3", T=1024, H=512, I=256, E=8, k=2, fmt="e4m3", zipf_bias=True),
    "wide_e2m1": W.custom("wide_e2m1", T=700, H=256, I=384, E=4, k=1, fmt="e2m1"),
    # degenerate shapes: one token; a single routed expert; k = E
    "one_token": W.custom("one_token", T=1, H=256, I=128, E=4, k=2, fmt="e4m3"),
    "one_expert": W.custom("one_expert", T=5, H=128, I=128, E=1, k=1, fmt="e2m1"),
    "k_equals_e": W.custom("k_equals_e", T=9, H=256, I=256, E=4, k=4, fmt="e4m3"),
    # wide schedule as CTA pairs in both GEMMs (every pair tile has four weight
    # row blocks), skewed experts: many token tiles, one partial tile, a few rows
    "pair_e4m3": W.custom("pair_e4m3", T=1500, H=512, I=512, E=16, k=4, fmt="e4m3", zipf_bias=True),
    "pair_e2m1": W.custom("pair_e2m1", T=900, H=1024, I=256, E=6, k=2, fmt="e2m1", zipf_bias=True),
    # the routing limits: 1024 routed experts (+1 shared), top-32
    "max_routing": W.custom("max_routing", T=40, H=128, I=128, E=1024, k=32, fmt="e2m1"),
}


@pytest.mark.parametrize("name", list(LAYER_CASES))
def test_layer_parity(name):
    wl = LAYER_CASES[name]
    L = build_layer(wl)
    # weights: GPU quantiser vs oracle quantiser, bit-exact
    for e in range(wl.E + 1):
        assert np.array_equal(L.w1c[e].cpu().numpy(), L.o1c[e]), f"W1 codes expert {e}"
        assert np.array_equal(L.w1s[e].cpu().numpy(), L.o1s[e]), f"W1 scales expert {e}"
        assert np.array_equal(L.w2c[e].cpu().numpy(), L.o2c[e]), f"W2 codes expert {e}"
        assert np.array_equal(L.w2s[e].cpu().numpy(), L.o2s[e]), f"W2 scales expert {e}"
    ref = oracle_forward(L, want_h=True)
    r = _steps(L)
    assert r["status"] == (0, 0)
    assert np.array_equal(r["act_c"].cpu().numpy(), ref["act_codes"])
    assert np.array_equal(r["act_s"].cpu().numpy(), ref["act_scales"])
    assert np.array_equal(r["ids"].cpu().numpy(), ref["ids"])
    np.testing.assert_allclose(r["w"].cpu().numpy(), ref["topk_w"], rtol=2e-6, atol=1e-7)
    rc, ro, rs = oracle.permute(ref["ids"], wl.E)
    assert np.array_equal(r["counts"].cpu().numpy(), rc)
    assert np.array_equal(r["offsets"].cpu().numpy(), ro)
    assert np.array_equal(r["ss"].cpu().numpy(), rs)
    frac, hrel = _check_h(r, ref, wl.I)
    print(f"h codes {name}: mismatch fraction {frac:.2e}, decoded rel L2 {hrel:.2e}")
    assert frac < 0.005 and hrel < 0.01, (frac, hrel)
    rel, mabs = out_errors(r["out"].double().cpu().numpy(), ref["out"])
    assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (rel, mabs)
    # the fused single call gives the same layer
    out = L.layer.forward(L.x, L.logits)
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    rel2, mabs2 = out_errors(out.double().cpu().numpy(), ref["out"])
    assert rel2 <= OUT_REL_L2 and mabs2 <= OUT_MAX_ABS_OVER_RMS, (rel2, mabs2)
    step_vs_fused = (out - r["out"]).abs().max().item() / max(r["out"].abs().max().item(), 1e-30)
    assert step_vs_fused < 1e-5


def test_prefill_full_size_sampled():
    """8192-token prefill workload at full size, in the launch configuration the
    benchmark times; the oracle evaluates a sample of tokens one by one."""
    wl = W.WORKLOADS["prefill_mxfp8"]
    logits, _ = W.draw_router_and_activations(wl, 0, "cuda")
    rng = np.random.default_rng(0)
    tokens = sorted(set([0, wl.T - 1] + rng.choice(wl.T, 14, replace=False).tolist()))
    rid, _ = oracle.route_topk(logits.cpu().numpy(), wl.k)
    need = set(int(e) for e in rid[tokens].ravel()) | {wl.E}
    L = build_layer(wl, oracle_experts=need)
    for e in sorted(need)[:4]:
        assert np.array_equal(L.w1c[e].cpu().numpy(), L.o1c[e])
        assert np.array_equal(L.w2c[e].cpu().numpy(), L.o2c[e])
    ref = oracle_forward(L, tokens=tokens)
    out = L.layer.forward(L.x, L.logits)
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    got = out[tokens].double().cpu().numpy()
    rel, mabs = out_errors(got, ref["out"])
    assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (rel, mabs)
    # bit-exact routing and permutation over the whole workload
    assert np.array_equal(ref["ids"], rid)
    r = _steps(L)
    assert np.array_equal(r["ids"].cpu().numpy(), rid)
    rc, ro, rs = oracle.permute(rid, wl.E)
    assert np.array_equal(r["offsets"].cpu().numpy(), ro)
    assert np.array_equal(r["ss"].cpu().numpy(), rs)
    assert np.array_equal(r["act_c"].cpu().numpy(), ref["act_codes"])
    # every token row is finite and the whole-layer output equals the step chain
    assert torch.isfinite(out).all()
    assert (out - r["out"]).abs().max().item() <= 1e-5 * r["out"].abs().max().item()


def test_zero_tokens_is_a_noop():
    wl = W.custom("empty", T=0, H=256, I=128, E=8, k=2)
    ws = mx.alloc_workspace(1024)
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    logits = torch.empty(0, 8, device="cuda")
    out = torch.empty(0, 256, device="cuda")
    w = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    mx.moe_forward(x, logits, w, w, "e4m3", wl.I, wl.k, out, ws)
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["decode_mxfp8", "ragged_e2m1"])
def test_forward_graph_capture(name):
    """moe_forward issues only kernel launches (no host synchronisation, no
    memset or allocation), so it can be captured in a CUDA graph and replayed;
    the replay gives the eager result."""
    wl = LAYER_CASES[name]
    L = build_layer(wl, oracle_experts="none")
    eager = L.layer.forward(L.x, L.logits).clone()
    out = torch.empty_like(eager)
    L.layer.forward(L.x, L.logits, out)           # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            L.layer.forward(L.x, L.logits, out)
    torch.cuda.current_stream().wait_stream(s)
    out.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    err = (out - eager).abs().max().item() / eager.abs().max().item()
    assert err < 1e-5, err


@pytest.mark.parametrize("name", ["ragged_e4m3", "wide_e4m3", "wide_e2m1", "pair_e4m3"])
def test_large_batch_prologue_matches_separate_launches(name, monkeypatch):
    """Batches above one permutation chunk (or on the wide schedule): the
    one-launch prologue (grid barriers between routing, counting, scatter and
    row gather) gives the layer of the separate permutation and gather
    launches, and the oracle's."""
    wl = LAYER_CASES[name]
    L = build_layer(wl)
    assert mx.moe_forward_launches(wl.T, wl.H, wl.I, wl.E, wl.k, wl.fmt) == 3
    ref = oracle_forward(L)
    one = L.layer.forward(L.x, L.logits).clone()
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    monkeypatch.setenv("MXMOE_SEPARATE_PERMUTE", "1")
    assert mx.moe_forward_launches(wl.T, wl.H, wl.I, wl.E, wl.k, wl.fmt) > 3
    sep = L.layer.forward(L.x, L.logits)
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    for got in (one, sep):
        rel, mabs = out_errors(got.double().cpu().numpy(), ref["out"])
        assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (rel, mabs)
    diff = (one - sep).abs().max().item() / sep.abs().max().item()
    assert diff < 1e-5, diff


@pytest.mark.parametrize("name,kps", [("tiny", "2"), ("decode_mxfp8", "2"), ("decode_mxfp4", "1")])
def test_layer_parity_other_stage_shape(name, kps, monkeypatch):
    """The narrow schedule with the other number of K chunks per pipeline stage."""
    monkeypatch.setenv("MXMOE_KPS", kps)
    wl = LAYER_CASES[name]
    L = build_layer(wl)
    ref = oracle_forward(L)
    out = L.layer.forward(L.x, L.logits)
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    rel, mabs = out_errors(out.double().cpu().numpy(), ref["out"])
    assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (rel, mabs)


@pytest.mark.parametrize("name,bn", [("wide_e4m3", "96"), ("wide_e4m3", "224"), ("wide_e2m1", "128"),
                                     ("wide_e2m1", "160"), ("decode_mxfp8", "64"), ("ragged_e4m3", "192"),
                                     ("decode_mxfp4", "32"), ("ragged_e2m1", "16")])
def test_layer_parity_other_tile_width(name, bn, monkeypatch):
    """Other token-tile widths than the shape's default: two accumulator buffers
    (96), one buffer with one or two K chunks per stage (128 .. 224), the gather4
    schedule at 16, 32 and 64 rows, and a wide tile on a shape whose experts hold
    few rows."""
    monkeypatch.setenv("MXMOE_BN", bn)
    wl = LAYER_CASES[name]
    L = build_layer(wl)
    ref = oracle_forward(L)
    out = L.layer.forward(L.x, L.logits)
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    rel, mabs = out_errors(out.double().cpu().numpy(), ref["out"])
    assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (rel, mabs)


@pytest.mark.parametrize("name,groups", [("wide_e4m3", "2"), ("ragged_e4m3", "1"), ("decode_mxfp8", "4")])
def test_layer_parity_down_tile_groups(name, groups, monkeypatch):
    """The down GEMM with its weight tiles split into groups run one after the
    other (the order the wide schedule uses so that the combine's atomics land on
    an L2-sized slice of `out`)."""
    monkeypatch.setenv("MXMOE_MGROUPS", groups)
    wl = LAYER_CASES[name]
    L = build_layer(wl)
    ref = oracle_forward(L)
    out = L.layer.forward(L.x, L.logits)
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    rel, mabs = out_errors(out.double().cpu().numpy(), ref["out"])
    assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (rel, mabs)


@pytest.mark.parametrize("name,bn", [("pair_e4m3", None), ("pair_e2m1", None), ("wide_e4m3", "128"),
                                     ("pair_e4m3", "96"), ("pair_e4m3", "224")])
def test_pair_schedule_matches_single_cta(name, bn, monkeypatch):
    """The wide schedule run as CTA pairs (M = 256 MMAs over two SMs, on
    request) and as single CTAs gives the same layer, and both match the
    oracle."""
    if bn:
        monkeypatch.setenv("MXMOE_BN", bn)
    wl = LAYER_CASES[name]
    L = build_layer(wl)
    ref = oracle_forward(L)
    outs = {}
    for pair in ("1", "0"):
        monkeypatch.setenv("MXMOE_PAIR", pair)
        out = L.layer.forward(L.x, L.logits)
        assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
        rel, mabs = out_errors(out.double().cpu().numpy(), ref["out"])
        assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (pair, rel, mabs)
        outs[pair] = out
    diff = (outs["1"] - outs["0"]).abs().max().item() / outs["0"].abs().max().item()
    assert diff < 1e-5, diff



# ------------------------------------------------------------------ layer variants
# SwiGLU-OAI: a clamp limit below the typical |g| of each shape (g ~ N(0, 0.02^2 H)
# for these weights) so that the clamp acts; specverify with a limit that does not
OAI_CASES = [("tiny", 0.2), ("decode_mxfp8", 0.7), ("ragged_e2m1", 0.3), ("wide_e4m3", 0.3),
             ("specverify_mxfp4", 7.0)]


@pytest.mark.parametrize("name,limit", OAI_CASES)
def test_swiglu_oai_layer_parity(name, limit):
    """The SwiGLU-OAI epilogue (caller alpha and clamp limit) against the
    oracle's: h codes within the one-step rules, the layer output within the
    output tolerance, through the step-wise call and the fused one."""
    alpha = 1.702
    wl = LAYER_CASES[name]
    L = build_layer(wl)
    ref = oracle.moe_forward(L.x_bits, L.logits_np, wl.k, L.o1c, L.o1s, L.o2c, L.o2s, L.fmt, wl.I, want_h=True,
                             act=oracle.ACT_SWIGLU_OAI, alpha=alpha, limit=limit)
    opts = mx.layer_opts("swiglu_oai", alpha=alpha, limit=limit)
    r = _steps(L, opts)
    assert r["status"] == (0, 0)
    frac, hrel = _check_h(r, ref, wl.I)
    print(f"h codes (SwiGLU-OAI) {name}: mismatch fraction {frac:.2e}, decoded rel L2 {hrel:.2e}")
    assert frac < 0.005 and hrel < 0.01, (frac, hrel)
    rel, mabs = out_errors(r["out"].double().cpu().numpy(), ref["out"])
    assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (rel, mabs)
    out = L.layer.forward(L.x, L.logits, opts=opts)
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    rel2, mabs2 = out_errors(out.double().cpu().numpy(), ref["out"])
    assert rel2 <= OUT_REL_L2 and mabs2 <= OUT_MAX_ABS_OVER_RMS, (rel2, mabs2)
    # the variant differs from the standard layer (the options reach the kernel)
    std = oracle_forward(L)["out"]
    assert np.linalg.norm(ref["out"] - std) > 10 * OUT_REL_L2 * np.linalg.norm(std)


@pytest.mark.parametrize("name", ["tiny", "decode_mxfp8", "specverify_mxfp4", "ragged_e4m3", "wide_e2m1",
                                  "max_routing"])
def test_dense_shared_expert_matches_folded(name):
    """The shared expert run as its own dense launches (the path the folded
    table replaces) gives the folded layer's output, and the oracle's."""
    wl = LAYER_CASES[name]
    L = build_layer(wl)
    ref = oracle_forward(L)
    folded = L.layer.forward(L.x, L.logits).clone()
    dense = L.layer.forward(L.x, L.logits, opts=mx.layer_opts(shared="dense"))
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    rel, mabs = out_errors(dense.double().cpu().numpy(), ref["out"])
    assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (rel, mabs)
    diff = (dense - folded).abs().max().item() / folded.abs().max().item()
    assert diff < 1e-5, diff


def test_dense_shared_expert_with_swiglu_oai():
    wl = LAYER_CASES["ragged_e4m3"]
    L = build_layer(wl)
    ref = oracle.moe_forward(L.x_bits, L.logits_np, wl.k, L.o1c, L.o1s, L.o2c, L.o2s, L.fmt, wl.I,
                             act=oracle.ACT_SWIGLU_OAI, alpha=1.5, limit=0.4)
    out = L.layer.forward(L.x, L.logits, opts=mx.layer_opts("swiglu_oai", alpha=1.5, limit=0.4, shared="dense"))
    assert mx.moe_get_status(L.layer.workspace(wl.T)) == 0
    rel, mabs = out_errors(out.double().cpu().numpy(), ref["out"])
    assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (rel, mabs)


# ---- MXFP4 activations (kind::mxf4: both operands packed E2M1)
@pytest.mark.parametrize("T,H", [(1, 32), (16, 256), (37, 4096), (6, 2048), (4096, 4096)])
def test_quantize_act_e2m1_bitexact(T, H):
    """x bf16 -> MXFP4 codes (two per byte, element 2i low) and E8M0 scales,
    bit-exact against the oracle's quantiser (emax 2, RNE, saturate at 6);
    special blocks as in the MXFP8 case."""
    x = _bf16(T, H, 11)
    if T >= 16:
        x[0, :32] = 0.0
        x[1, :32] = -0.0
        x[2, :32] = 1e-39
        x[3, :32] = 3.0e38
    codes = torch.empty(T, H // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(T, H // 32, dtype=torch.uint8, device="cuda")
    mx.mx_quantize_act(x.cuda(), codes, scales, fmt="e2m1")
    rc, rs = oracle.quantize_bf16(W.bf16_bits(x), oracle.E2M1)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def _nibbles(c):
    c = c.astype(np.int64)
    return np.stack([c & 15, c >> 4], axis=-1).reshape(c.shape[0], -1)


A4_CASES = ["decode_mxfp4", "specverify_mxfp4", "ragged_e2m1", "wide_e2m1", "one_expert", "max_routing"]


@pytest.mark.parametrize("name", A4_CASES)
def test_mxfp4_activations_layer_parity(name):
    """MXFP4 activations and h on the packed-FP4 MMA against the oracle run
    with the same MXFP4 quantisation of x and h: activation codes bit-exact,
    h codes equal but for rare one-step flips at rounding boundaries, the
    layer output within the same tolerance as the MXFP8 layer (the oracle does
    the same quantisations; the GPU accumulates in fp32).  The variant's output
    differs from the MXFP8-activation layer by far more than that tolerance."""
    wl = LAYER_CASES[name]
    L = build_layer(wl)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    ref = oracle.moe_forward(L.x_bits, L.logits_np, k, L.o1c, L.o1s, L.o2c, L.o2s, L.fmt, I, want_h=True,
                             act_fmt=oracle.E2M1)
    opts = mx.layer_opts(act_fmt="e2m1")
    # step-wise calls
    act_c = torch.empty(T, H // 2, dtype=torch.uint8, device="cuda")
    act_s = torch.empty(T, H // 32, dtype=torch.uint8, device="cuda")
    mx.mx_quantize_act(L.x, act_c, act_s, fmt="e2m1")
    assert np.array_equal(act_c.cpu().numpy(), ref["act_codes"])
    assert np.array_equal(act_s.cpu().numpy(), ref["act_scales"])
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    mx.moe_route_topk(L.logits, k, ids, w)
    counts = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 2, dtype=torch.int32, device="cuda")
    ss = torch.empty(T * (k + 1), dtype=torch.int32, device="cuda")
    pws = mx.alloc_workspace(mx.moe_permute_workspace_size(T, E, k))
    mx.moe_permute(ids, E, counts, offsets, ss, pws)
    gws = mx.alloc_workspace(mx.moe_gemm_workspace_size(T, H, I, E, k))
    h_c = torch.empty(T * (k + 1), I // 2, dtype=torch.uint8, device="cuda")
    h_s = torch.empty(T * (k + 1), I // 32, dtype=torch.uint8, device="cuda")
    mx.moe_grouped_gemm_swiglu_ex(act_c, act_s, offsets, ss, L.layer.w1, L.fmt, T, H, I, E, k, h_c, h_s, gws, opts)
    out = torch.zeros(T, H, dtype=torch.float32, device="cuda")
    mx.moe_grouped_gemm_down_combine(h_c, h_s, offsets, ss, w, L.layer.w2, L.fmt, T, H, I, E, k, out, gws, opts=opts)
    assert (mx.moe_get_status(pws), mx.moe_get_status(gws)) == (0, 0)
    srt = ss.cpu().numpy()
    gc, gs = h_c.cpu().numpy(), h_s.cpu().numpy()
    rc, rs = ref["h_codes"][srt], ref["h_scales"][srt]
    assert np.all(np.abs(gs.astype(np.int64) - rs.astype(np.int64)) <= 1), "a block scale moved by more than one"
    gv = oracle.decode_matrix(gc, gs, oracle.E2M1)
    rv = oracle.decode_matrix(rc, rs, oracle.E2M1)
    frac = np.count_nonzero(_nibbles(gc) != _nibbles(rc)) / (gc.size * 2)
    hrel = np.linalg.norm(gv - rv) / np.linalg.norm(rv)
    print(f"MXFP4 h codes {name}: mismatch fraction {frac:.2e}, decoded rel L2 {hrel:.2e}")
    assert frac < 0.005 and hrel < 0.02, (frac, hrel)
    rel, mabs = out_errors(out.double().cpu().numpy(), ref["out"])
    assert rel <= OUT_REL_L2 and mabs <= OUT_MAX_ABS_OVER_RMS, (rel, mabs)
    # the fused single call
    fused = L.layer.forward(L.x, L.logits, opts=opts)
    assert mx.moe_get_status(L.layer.workspace(T)) == 0
    rel2, mabs2 = out_errors(fused.double().cpu().numpy(), ref["out"])
    assert rel2 <= OUT_REL_L2 and mabs2 <= OUT_MAX_ABS_OVER_RMS, (rel2, mabs2)
    # a different layer from the MXFP8-activation one
    std = oracle_forward(L)["out"]
    assert np.linalg.norm(ref["out"] - std) > 4 * OUT_REL_L2 * np.linalg.norm(std)


@pytest.mark.parametrize("name", ["tiny", "wide_e4m3"])
def test_gemm_launch_timing_hook(name):
    """mx_debug_time_gemms brackets each grouped-GEMM launch with events: the
    step-wise layer records one gate/up and one down launch with positive
    device times (the wide schedule's row gather is not inside them), reading
    clears them, and nothing is recorded while timing is off."""
    wl = LAYER_CASES[name]
    L = build_layer(wl)
    mx.mx_debug_time_gemms(True)
    try:
        r = _steps(L)
        torch.cuda.synchronize()
        ms, epi = mx.mx_debug_gemm_times()
        assert epi == [0, 1], epi
        assert all(0.0 < t < 1000.0 for t in ms), ms
        assert mx.mx_debug_gemm_times() == ([], [])
    finally:
        mx.mx_debug_time_gemms(False)
    assert r["status"] == (0, 0)
    _steps(L)
    torch.cuda.synchronize()
    assert mx.mx_debug_gemm_times() == ([], [])
