"""Pins for the oracle's router, permutation and expert layer against library
routines and identities: numpy's stable argsort (top-k order with lowest-index
tie-break, expert grouping), scipy's softmax, routed-count invariants, an
independent numpy formulation of the layer (per-token loops, BLAS matmuls,
scipy's logistic function), the folded-shared-expert == separate dense SwiGLU
MLP identity, exact integer arithmetic on tiny inputs, and the k = E average."""
import numpy as np
import pytest
import scipy.special as sps


def _logits(rng, T, E, ties=False):
    if ties:
        return rng.integers(-3, 4, size=(T, E)).astype(np.float32)
    return rng.standard_normal((T, E)).astype(np.float32)


@pytest.mark.parametrize("T,E,k,ties", [(5, 8, 2, False), (17, 16, 4, True), (3, 6, 6, True), (40, 32, 8, False)])
def test_topk_matches_stable_argsort(orc, T, E, k, ties):
    rng = np.random.default_rng(T * 100 + E)
    l = _logits(rng, T, E, ties)
    ids, w = orc.route_topk(l, k)
    ref = np.argsort(-l, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref)
    sel = np.take_along_axis(l.astype(np.float64), ids, axis=1)
    assert np.allclose(w, sps.softmax(sel, axis=1), rtol=1e-14, atol=0)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)
    # ratios fixed by the logit differences
    assert np.allclose(w[:, 0] / w[:, -1], np.exp(sel[:, 0] - sel[:, -1]), rtol=1e-12)
    # ids distinct per token
    assert all(len(set(r)) == k for r in ids.tolist())


def test_topk_tie_takes_lowest_index(orc):
    l = np.zeros((1, 6), dtype=np.float32)
    l[0, [1, 3, 4]] = 2.0
    ids, w = orc.route_topk(l, 4)
    assert ids.tolist() == [[1, 3, 4, 0]]


def test_softmax_over_selected_equals_renormalised_full_softmax(orc):
    rng = np.random.default_rng(1)
    l = _logits(rng, 9, 12)
    ids, w = orc.route_topk(l, 3)
    full = sps.softmax(l.astype(np.float64), axis=1)
    sel = np.take_along_axis(full, ids, axis=1)
    assert np.allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-13)


@pytest.mark.parametrize("T,E,k", [(7, 5, 2), (33, 16, 4), (1, 4, 4), (64, 128, 8)])
def test_permute_invariants_and_stable_sort(orc, T, E, k):
    rng = np.random.default_rng(T + E + k)
    ids, _ = orc.route_topk(_logits(rng, T, E, ties=True), k)
    counts, offsets, ss = orc.permute(ids, E)
    assert counts[:E].sum() == T * k and counts[E] == T
    assert offsets[0] == 0 and offsets[-1] == T * (k + 1)
    assert np.all(np.diff(offsets) == counts)
    assert sorted(ss.tolist()) == list(range(T * (k + 1)))
    # library formulation: stable sort of slot ids by their expert (shared = E)
    ex = np.concatenate([ids, np.full((T, 1), E, dtype=np.int32)], axis=1).ravel()
    assert np.array_equal(ss, np.argsort(ex, kind="stable"))
    for e in range(E + 1):
        seg = ss[offsets[e]:offsets[e + 1]]
        assert np.all(ex[seg] == e)
        assert np.all(np.diff(seg // (k + 1)) > 0)


# ---------------------------------------------------------------- router GEMM + biased top-k
def _bf16_bits(a):
    """fp32 array -> bf16 bit patterns (round to nearest even) and the exact values."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16), t.double().numpy()


def test_router_logits_exact_on_integers_and_match_blas(orc):
    """Small integers are exact in bf16 and their dot products exact in fp64:
    the logits equal integer matmul; on random inputs they equal a BLAS fp64
    matmul of the same bf16 values to rounding."""
    rng = np.random.default_rng(3)
    xi = rng.integers(-8, 9, size=(5, 96))
    wi = rng.integers(-8, 9, size=(7, 96))
    xb, _ = _bf16_bits(xi)
    wb, _ = _bf16_bits(wi)
    assert np.array_equal(orc.router_logits(xb, wb), (xi @ wi.T).astype(np.float64))
    xb, xv = _bf16_bits(rng.standard_normal((9, 256)))
    wb, wv = _bf16_bits(rng.standard_normal((12, 256)) * 0.05)
    got = orc.router_logits(xb, wb)
    assert got.shape == (9, 12)
    assert np.allclose(got, xv @ wv.T, rtol=1e-12, atol=1e-12)


def test_biased_topk(orc):
    """A zero bias is plain top-k; a dominating bias forces its expert into
    every token's selection while the weights stay the softmax of the chosen
    experts' unbiased logits; brute force on fp32 scores with ties."""
    rng = np.random.default_rng(8)
    l = rng.standard_normal((20, 16)).astype(np.float32)
    ids0, w0 = orc.route_topk(l, 4)
    ids1, w1 = orc.route_topk_biased(l, np.zeros(16, np.float32), 4)
    assert np.array_equal(ids0, ids1) and np.array_equal(w0, w1)
    ids_n, _ = orc.route_topk_biased(l, None, 4)
    assert np.array_equal(ids_n, ids0)
    bias = np.zeros(16, np.float32)
    bias[11] = 100.0
    ids, w = orc.route_topk_biased(l, bias, 4)
    assert np.all(ids[:, 0] == 11)
    for t in range(20):
        sel = l[t, ids[t]].astype(np.float64)
        assert np.allclose(w[t], sps.softmax(sel), rtol=1e-14)
        rest = np.setdiff1d(np.arange(16), ids[t])
        assert np.min((l[t] + bias)[ids[t]]) >= np.max((l[t] + bias)[rest])
    # ties in the biased score resolve to the lowest index
    lt = rng.integers(-2, 3, size=(30, 10)).astype(np.float32)
    bt = rng.integers(-1, 2, size=10).astype(np.float32)
    ids, _ = orc.route_topk_biased(lt, bt, 5)
    score = (lt + bt).astype(np.float32)
    want = np.argsort(-score, axis=1, kind="stable")[:, :5]
    assert np.array_equal(ids, want)


# ---------------------------------------------------------------- expert layer
def _random_layer(orc, rng, T, H, I, E, k, fmt, std=0.05, act_fmt=None):
    w1c, w1s, w2c, w2s = [], [], [], []
    for _ in range(E + 1):
        c, s = orc.quantize_rows(rng.standard_normal((2 * I, H)) * std, fmt)
        w1c.append(c), w1s.append(s)
        c, s = orc.quantize_rows(rng.standard_normal((H, I)) * std, fmt)
        w2c.append(c), w2s.append(s)
    x = rng.standard_normal((T, H))
    act_c, act_s = orc.quantize_rows(x, orc.E4M3 if act_fmt is None else act_fmt)
    l = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = orc.route_topk(l, k)
    return act_c, act_s, ids, w, w1c, w1s, w2c, w2s


def _numpy_layer(orc, act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I, requant=True, skip_shared=False,
                 oai=None, act_fmt=None):
    """Per-token loops with no permutation: BLAS matmuls, scipy's logistic.
    oai = (alpha, limit): the SwiGLU-OAI activation; act_fmt: the MX format of
    the activations and of h (default MXFP8)."""
    act_fmt = orc.E4M3 if act_fmt is None else act_fmt
    T = act_c.shape[0]
    H = act_s.shape[1] * 32
    E = len(w1c) - 1
    k = ids.shape[1]
    x = orc.decode_matrix(act_c, act_s, act_fmt)
    out = np.zeros((T, H))
    dec1 = [orc.decode_matrix(w1c[e], w1s[e], fmt) for e in range(E + 1)]
    dec2 = [orc.decode_matrix(w2c[e], w2s[e], fmt) for e in range(E + 1)]
    for t in range(T):
        pairs = [(int(ids[t, j]), w[t, j]) for j in range(k)]
        if not skip_shared:
            pairs.append((E, 1.0))
        for e, wt in pairs:
            g = dec1[e][:I] @ x[t]
            u = dec1[e][I:] @ x[t]
            if oai is None:
                h = g * sps.expit(g) * u
            else:
                alpha, limit = oai
                gc, uc = np.minimum(g, limit), np.clip(u, -limit, limit)
                h = gc * sps.expit(alpha * gc) * (uc + 1.0)
            if requant:
                hc, hs = orc.quantize_rows(h[None, :], act_fmt)
                h = orc.decode_matrix(hc, hs, act_fmt)[0]
            out[t] += wt * (dec2[e] @ h)
    return out


@pytest.mark.parametrize("fmt_name,T,H,I,E,k", [("e4m3", 6, 64, 32, 4, 2), ("e2m1", 5, 64, 64, 6, 3)])
def test_layer_matches_numpy_per_token_loops(orc, fmt_name, T, H, I, E, k):
    fmt = orc.E4M3 if fmt_name == "e4m3" else orc.E2M1
    rng = np.random.default_rng(11)
    act_c, act_s, ids, w, w1c, w1s, w2c, w2s = _random_layer(orc, rng, T, H, I, E, k, fmt)
    res = orc.expert_layer(act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I, want_noq=True, want_h=True)
    ref = _numpy_layer(orc, act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I)
    scale = np.sqrt(np.mean(ref ** 2))
    assert np.max(np.abs(res["out"] - ref)) <= 1e-12 * scale
    ref_noq = _numpy_layer(orc, act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I, requant=False)
    assert np.max(np.abs(res["out_noq"] - ref_noq)) <= 1e-12 * scale
    # requantised h differs from unquantised h by about one E4M3 step (2^-4 relative)
    rel = np.linalg.norm(res["out"] - res["out_noq"]) / np.linalg.norm(res["out_noq"])
    assert 1e-4 < rel < 5e-2
    # token subset gives the same rows
    sub = orc.expert_layer(act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I, tokens=[4, 0, 2])
    assert np.array_equal(sub["out"], res["out"][[4, 0, 2]])


def test_swiglu_oai_special_cases(orc):
    """SwiGLU-OAI against textbook functions where it reduces to one: a clamp
    limit of 0 leaves silu of the non-positive part of the gate (the up
    projection clamps to 0 and enters as 0 + 1); alpha = 1 with no clamp is
    silu(g) * (u + 1); a steep sigmoid is relu(g) * (u + 1); clamping caps the
    gate from above only and the up projection on both sides."""
    g = np.linspace(-6, 6, 49)
    u = np.linspace(3, -3, 49)
    silu = g * sps.expit(g)
    assert np.allclose(orc.swiglu_oai(g, u, 1.0, 0.0), np.where(g < 0, silu, 0.0), rtol=1e-14, atol=1e-15)
    assert np.allclose(orc.swiglu_oai(g, u, 1.0, np.inf), silu * (u + 1.0), rtol=1e-14, atol=1e-15)
    steep = orc.swiglu_oai(g[np.abs(g) > 1], u[np.abs(g) > 1], 200.0, np.inf)
    assert np.allclose(steep, np.maximum(g, 0)[np.abs(g) > 1] * (u[np.abs(g) > 1] + 1.0), rtol=1e-12, atol=1e-12)
    # gate 10 and up -10 under a limit of 7: 7 * sigmoid(1.702 * 7) * (-7 + 1)
    assert np.isclose(orc.swiglu_oai([10.0], [-10.0], 1.702, 7.0)[0], 7.0 * sps.expit(1.702 * 7.0) * -6.0, rtol=1e-14)
    # a gate far below the limit is left alone
    assert np.isclose(orc.swiglu_oai([-10.0], [0.5], 1.0, 7.0)[0], -10.0 * sps.expit(-10.0) * 1.5, rtol=1e-14)


@pytest.mark.parametrize("variant", ["oai_e4m3", "swiglu_e2m1_act", "oai_e2m1_act"])
def test_layer_variants_match_numpy_per_token_loops(orc, variant):
    """The layer with the SwiGLU-OAI activation and/or MXFP4 activations (and
    MXFP4 h) against the per-token formulation, with a clamp limit small enough
    that part of g and u is clamped."""
    rng = np.random.default_rng(23)
    T, H, I, E, k = 6, 64, 64, 5, 2
    oai = (1.702, 0.15) if variant.startswith("oai") else None
    fp4 = variant.endswith("e2m1_act")
    fmt = orc.E2M1 if fp4 else orc.E4M3
    act_fmt = orc.E2M1 if fp4 else orc.E4M3
    act_c, act_s, ids, w, w1c, w1s, w2c, w2s = _random_layer(orc, rng, T, H, I, E, k, fmt, std=0.1, act_fmt=act_fmt)
    kw = dict(act_fmt=act_fmt)
    if oai:
        kw.update(act=orc.ACT_SWIGLU_OAI, alpha=oai[0], limit=oai[1])
    res = orc.expert_layer(act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I, want_noq=True, want_h=True, **kw)
    ref = _numpy_layer(orc, act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I, oai=oai, act_fmt=act_fmt)
    scale = np.sqrt(np.mean(ref ** 2))
    assert scale > 0
    assert np.max(np.abs(res["out"] - ref)) <= 1e-12 * scale
    ref_noq = _numpy_layer(orc, act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I, requant=False, oai=oai,
                           act_fmt=act_fmt)
    assert np.max(np.abs(res["out_noq"] - ref_noq)) <= 1e-12 * scale
    assert res["h_codes"].shape[1] == (I // 2 if fp4 else I)
    if oai:
        # the clamp is active: some gate values exceed the limit
        x = orc.decode_matrix(act_c, act_s, act_fmt)
        g = x @ orc.decode_matrix(w1c[E], w1s[E], fmt)[:I].T
        assert np.any(g > oai[1]) and np.any(g < oai[1])


def test_folded_shared_expert_equals_separate_dense_mlp(orc):
    """Folding the shared expert into the routed table as an always-selected
    slot of weight 1 gives the routed-only layer plus a dense SwiGLU MLP."""
    rng = np.random.default_rng(5)
    T, H, I, E, k, fmt = 7, 64, 32, 5, 2, orc.E4M3
    act_c, act_s, ids, w, w1c, w1s, w2c, w2s = _random_layer(orc, rng, T, H, I, E, k, fmt)
    full = orc.expert_layer(act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I)["out"]
    # routed only: the shared expert's down projection zeroed
    w2c0 = list(w2c)
    w2c0[E] = np.zeros_like(w2c[E])
    routed = orc.expert_layer(act_c, act_s, ids, w, w1c, w1s, w2c0, w2s, fmt, I)["out"]
    x = orc.decode_matrix(act_c, act_s, orc.E4M3)
    W1 = orc.decode_matrix(w1c[E], w1s[E], fmt)
    W2 = orc.decode_matrix(w2c[E], w2s[E], fmt)
    g, u = x @ W1[:I].T, x @ W1[I:].T
    h = g * sps.expit(g) * u
    hc, hs = orc.quantize_rows(h, orc.E4M3)
    dense = orc.decode_matrix(hc, hs, orc.E4M3) @ W2.T
    assert np.max(np.abs(full - (routed + dense))) <= 1e-12 * np.sqrt(np.mean(full ** 2))


def test_gemms_exact_on_integer_inputs(orc):
    """With small integer codes and unit scales every product and partial sum
    is an exact integer in fp64, so g and u equal exact integer arithmetic;
    weights of zero for the down projection except a one-hot row pick h_i."""
    rng = np.random.default_rng(9)
    T, H, I, E, k = 3, 32, 32, 1, 1
    ints = np.array([0x38, 0x40, 0x44, 0xB8, 0xC0, 0x00])   # 1, 2, 3, -1, -2, 0 in E4M3
    act_c = rng.choice(ints, size=(T, H)).astype(np.uint8)
    act_s = np.full((T, 1), 127, dtype=np.uint8)
    w1c = [rng.choice(ints, size=(2 * I, H)).astype(np.uint8) for _ in range(2)]
    w1s = [np.full((2 * I, 1), 127, dtype=np.uint8) for _ in range(2)]
    # down projection: output row o reads h_o (identity), scale 1
    eye = np.where(np.eye(H, I, dtype=bool), 0x38, 0x00).astype(np.uint8)
    w2c = [eye, np.zeros((H, I), dtype=np.uint8)]
    w2s = [np.full((H, 1), 127, dtype=np.uint8)] * 2
    ids = np.zeros((T, 1), dtype=np.int32)
    w = np.ones((T, 1))
    res = orc.expert_layer(act_c, act_s, ids, w, w1c, w1s, w2c, w2s, orc.E4M3, I, want_noq=True)
    val = {0x38: 1, 0x40: 2, 0x44: 3, 0xB8: -1, 0xC0: -2, 0x00: 0}
    X = np.vectorize(val.get)(act_c).astype(object)
    W = np.vectorize(val.get)(w1c[0]).astype(object)
    G = X.dot(W[:I].T)
    U = X.dot(W[I:].T)
    for t in range(T):
        for i in range(I):
            g, u = int(G[t, i]), int(U[t, i])
            assert res["out_noq"][t, i] == pytest.approx(g * sps.expit(g) * u, rel=1e-13, abs=1e-300)


def test_k_equals_e_equal_logits_is_dense_average(orc):
    rng = np.random.default_rng(4)
    T, H, I, E, k, fmt = 4, 32, 32, 4, 4, orc.E4M3
    act_c, act_s, _, _, w1c, w1s, w2c, w2s = _random_layer(orc, rng, T, H, I, E, k, fmt)
    ids, w = orc.route_topk(np.zeros((T, E), dtype=np.float32), k)
    assert np.array_equal(ids, np.tile(np.arange(E), (T, 1)))
    assert np.all(w == 0.25)
    res = orc.expert_layer(act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I)["out"]
    per = []
    for e in range(E + 1):
        ide = np.full((T, 1), min(e, E - 1), dtype=np.int32)
        one = _numpy_layer(orc, act_c, act_s, ide, np.ones((T, 1)), w1c, w1s, w2c, w2s, fmt, I,
                           skip_shared=True) if e < E else None
        per.append(one)
    x = orc.decode_matrix(act_c, act_s, orc.E4M3)
    W1 = orc.decode_matrix(w1c[E], w1s[E], fmt)
    W2 = orc.decode_matrix(w2c[E], w2s[E], fmt)
    g, u = x @ W1[:I].T, x @ W1[I:].T
    hc, hs = orc.quantize_rows(g * sps.expit(g) * u, orc.E4M3)
    shared = orc.decode_matrix(hc, hs, orc.E4M3) @ W2.T
    dense_avg = sum(per[:E]) / E + shared
    assert np.max(np.abs(res - dense_avg)) <= 1e-12 * np.sqrt(np.mean(res ** 2))


def test_layer_rejects_missing_expert(orc):
    rng = np.random.default_rng(2)
    T, H, I, E, k, fmt = 3, 32, 32, 3, 1, orc.E4M3
    act_c, act_s, ids, w, w1c, w1s, w2c, w2s = _random_layer(orc, rng, T, H, I, E, k, fmt)
    w1c = list(w1c)
    w1c[int(ids[0, 0])] = None
    with pytest.raises(ValueError):
        orc.expert_layer(act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, I)


def test_layer_result_does_not_depend_on_thread_count(orc):
    """Every output of the oracle is computed by one thread in index order, so
    one thread and all cores give bit-identical layers (the benchmark times both)."""
    rng = np.random.default_rng(5)
    fmt = orc.E4M3
    act_c, act_s, ids, w, w1c, w1s, w2c, w2s = _random_layer(orc, rng, 9, 64, 64, 6, 3, fmt)
    try:
        orc.set_threads(1)
        one = orc.expert_layer(act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, 64, want_h=True)
        orc.set_threads(0)
        many = orc.expert_layer(act_c, act_s, ids, w, w1c, w1s, w2c, w2s, fmt, 64, want_h=True)
    finally:
        orc.set_threads(0)
    assert np.array_equal(one["out"], many["out"])
    assert np.array_equal(one["h_codes"], many["h_codes"])
