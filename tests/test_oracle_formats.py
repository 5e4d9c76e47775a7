"""Pins for the oracle's MX codec (decode, block quantisation) against things
other than the oracle itself: torch's float8 dtypes (an independent library
implementation of E4M3 and E8M0), the OCP MX v1.0 E2M1 value table, hand-worked
blocks (tests/golden/mx_handworked.json) and brute-force nearest-value search."""
import json
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_handworked.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_e4m3_decode_matches_torch_float8(orc):
    codes = np.arange(256)
    ours = orc.decode_e4m3(codes)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign of zero
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def test_e8m0_decode_matches_torch(orc):
    ours = orc.decode_e8m0(np.arange(256))
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    assert np.isnan(ours[255]) and np.isnan(ref[255])
    assert np.array_equal(ours[:255], ref[:255])


def test_e2m1_decode_matches_spec_table(orc):
    mags = np.array(_golden()["e2m1_magnitudes"])
    ours = orc.decode_e2m1(np.arange(16))
    assert np.array_equal(ours[:8], mags)
    assert np.array_equal(ours[8:], -mags)
    assert np.signbit(ours[8])


@pytest.mark.parametrize("case", range(len(_golden()["blocks"])))
def test_handworked_blocks(orc, case):
    blk = _golden()["blocks"][case]
    fmt = orc.E4M3 if blk["fmt"] == "e4m3" else orc.E2M1
    v = np.zeros(32)
    for i, x in blk["values"].items():
        v[int(i)] = x
    codes, scale = orc.quantize_block(v, fmt)
    want = np.zeros(32, dtype=np.uint8)
    for i, c in blk["codes"].items():
        want[int(i)] = c
    assert scale == blk["scale"], blk["why"]
    assert np.array_equal(codes, want), (blk["why"], codes, want)


def _nearest_even(q, values, codes):
    """Brute force: nearest representable magnitude, ties to the even code,
    saturating at the largest finite value."""
    a = abs(q)
    d = np.abs(values - a)
    best = np.min(d)
    cand = codes[d == best]
    even = [c for c in cand if c % 2 == 0]
    return int(even[0] if even else cand[0])


@pytest.mark.parametrize("fmt_name", ["e4m3", "e2m1"])
def test_rounding_matches_brute_force(orc, fmt_name):
    rng = np.random.default_rng(7)
    if fmt_name == "e4m3":
        fmt, pin, signbit = orc.E4M3, 256.0, 0x80   # 256 fixes the block exponent at 0
        codes = np.arange(0x7F)
        vals = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
        grid = vals[vals > 0]
    else:
        fmt, pin, signbit = orc.E2M1, 7.9, 0x8     # 7.9 fixes the block exponent at 0
        codes = np.arange(8)
        vals = np.array(_golden()["e2m1_magnitudes"])
        grid = vals[vals > 0]
    for _ in range(60):
        v = np.empty(32)
        v[0] = pin
        # half the entries sit exactly on rounding midpoints, the rest anywhere
        mids = (grid[:-1] + grid[1:]) / 2
        n_mid = 15
        v[1:1 + n_mid] = rng.choice(np.concatenate([mids, grid[:1] / 2]), n_mid) * rng.choice([-1, 1], n_mid)
        v[1 + n_mid:] = rng.uniform(-pin, pin, 32 - 1 - n_mid)
        got, scale = orc.quantize_block(v, fmt)
        assert scale == 127
        for i in range(32):
            want = _nearest_even(v[i], vals, codes)
            if v[i] < 0 or (v[i] == 0 and np.signbit(v[i])):
                want |= signbit
            assert got[i] == want, (fmt_name, v[i], got[i], want)


def test_round_trip_every_code(orc):
    """decode(quantise(decode(c) * 2^s)) == c at a fixed block exponent s."""
    for fmt, maxcode, pin_code in ((orc.E4M3, 0x7E, 0x7E), (orc.E2M1, 0x7, 0x7)):
        dec = orc.decode_e4m3 if fmt == orc.E4M3 else orc.decode_e2m1
        signbit = 0x80 if fmt == orc.E4M3 else 0x8
        for s in (-20, 0, 9):
            allc = [c for c in range(maxcode + 1)] + [c | signbit for c in range(1, maxcode + 1)]
            for start in range(0, len(allc), 31):
                chunk = allc[start:start + 31]
                v = np.zeros(32)
                v[0] = float(dec([pin_code])[0]) * 2.0 ** s   # amax -> exponent s
                v[1:1 + len(chunk)] = dec(chunk) * 2.0 ** s
                got, sc = orc.quantize_block(v, fmt)
                assert sc == s + 127
                assert list(got[1:1 + len(chunk)]) == chunk


def test_activation_quantiser_matches_torch_fp8_cast(orc):
    """bf16 rows -> MXFP8, checked against torch.frexp (block exponent) and
    torch's fp32 -> float8_e4m3fn cast (RNE) where the value is in range."""
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(64, 256, generator=g) * torch.exp(torch.randn(64, 1, generator=g) * 4)).to(torch.bfloat16)
    x[0, :32] = 0.0
    x[1, 5] = 3.0e-39   # a bf16 subnormal in an otherwise normal block
    x[2, :32] = 1.0e-39  # an all-subnormal block
    codes, scales = orc.quantize_bf16(x.view(torch.int16).numpy().view(np.uint16))
    xf = x.double().view(64, 8, 32)
    amax = xf.abs().amax(-1)
    _, ex = torch.frexp(amax)
    s = torch.where(amax > 0, ex - 1 - 8, torch.full_like(ex, -127)).clamp(-127, 127)
    assert np.array_equal(scales, (s + 127).numpy().astype(np.uint8))
    q = (xf * torch.pow(2.0, -s.double())[..., None]).float()
    ref = q.to(torch.float8_e4m3fn).view(torch.uint8).view(64, 256).numpy().copy()
    over = (q.abs() > 448).view(64, 256).numpy()
    ref[over] = np.where(q.view(64, 256).numpy()[over] < 0, 0xFE, 0x7E)
    assert np.array_equal(codes, ref)


def test_e2m1_packing_low_nibble_first(orc):
    v = np.zeros((1, 32))
    v[0, 0], v[0, 1], v[0, 2] = 6.0, -0.5, 1.0
    codes, scales = orc.quantize_rows(v, orc.E2M1)
    assert codes.shape == (1, 16) and scales[0, 0] == 127
    assert codes[0, 0] == (0x7 | (0x9 << 4))
    assert codes[0, 1] == 0x2
    back = orc.decode_matrix(codes, scales, orc.E2M1)
    assert back[0, 0] == 6.0 and back[0, 1] == -0.5 and back[0, 2] == 1.0


def test_nonfinite_is_rejected(orc):
    v = np.zeros(32)
    v[3] = np.nan
    with pytest.raises(ValueError):
        orc.quantize_block(v, orc.E4M3)
    v[3] = np.inf
    with pytest.raises(ValueError):
        orc.quantize_block(v, orc.E2M1)


def _brute_force_mx(w64, grid, emax, signbit):
    """MX quantisation of fp64 rows written independently of the oracle: block
    exponent from numpy's frexp, elements divided by 2^exponent, nearest value
    of `grid` (the element format's non-negative magnitudes in code order) by
    exhaustive search, ties to the even code, sign kept."""
    rows, K = w64.shape
    blocks = w64.reshape(rows, K // 32, 32)
    amax = np.abs(blocks).max(-1)
    _, ex = np.frexp(amax)
    s = np.where(amax > 0, ex - 1 - emax, -127).clip(-127, 127)
    q = blocks * np.exp2(-s.astype(np.float64))[..., None]
    d = np.abs(np.abs(q)[..., None] - grid)            # [rows, K/32, 32, n_codes]
    best = d.min(-1, keepdims=True)
    cand = d == best
    n = grid.size
    # the lowest even code among the nearest, else the lowest code
    even = cand & (np.arange(n) % 2 == 0)
    code = np.where(even.any(-1), np.argmax(even, -1), np.argmax(cand, -1))
    code = code | np.where(np.signbit(q), signbit, 0)
    return code.reshape(rows, K).astype(np.uint8), (s + 127).astype(np.uint8)


@pytest.mark.parametrize("fmt_name", ["e4m3", "e2m1"])
def test_weight_quantiser_matches_brute_force(orc, fmt_name):
    """fp32 weight rows -> MX codes and scales, against a brute-force
    quantisation built from torch's E4M3 value table (or the OCP E2M1 table)
    and numpy's frexp.  The row count is odd and exceeds the oracle's thread
    count, and K = 96 is not a power of two, so a wrong row stride, a wrong row
    copy or a lost row in the parallel split shows up."""
    import os

    rows, K = 2 * (os.cpu_count() or 1) + 5, 96
    g = torch.Generator().manual_seed(11)
    w = torch.randn(rows, K, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 3) * 0.02
    w[0, :32] = 0.0
    w[1, 4] = -1e-30            # negative that rounds to -0 in its block
    w[2, 40] = 7.9 * 2.0 ** 3   # in the E2M1 saturation region of its block
    w[2, 41] = 1.0
    w = w.numpy()
    if fmt_name == "e4m3":
        fmt, emax, signbit = orc.E4M3, 8, 0x80
        grid = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    else:
        fmt, emax, signbit = orc.E2M1, 2, 0x8
        grid = np.array(_golden()["e2m1_magnitudes"])
    want_codes, want_scales = _brute_force_mx(w.astype(np.float64), grid, emax, signbit)
    codes, scales = orc.quantize_f32(w, fmt)
    assert np.array_equal(scales, want_scales)
    if fmt == orc.E2M1:
        assert codes.shape == (rows, K // 2)
        codes = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(rows, K)
    assert np.array_equal(codes, want_codes), np.argwhere(codes != want_codes)[:5]


@pytest.mark.parametrize("fmt_name", ["e4m3", "e2m1"])
def test_weight_quantiser_equals_row_quantiser(orc, fmt_name):
    """quantize_f32 (fp32 input, rows split over threads) gives the same bytes
    as quantize_rows on the same values widened to fp64, and rejects a
    non-finite entry in any row."""
    fmt = orc.E4M3 if fmt_name == "e4m3" else orc.E2M1
    rows, K = 3 * (os.cpu_count() or 1) + 1, 160
    w = (np.random.default_rng(5).standard_normal((rows, K)) * 0.02).astype(np.float32)
    c32, s32 = orc.quantize_f32(w, fmt)
    c64, s64 = orc.quantize_rows(w.astype(np.float64), fmt)
    assert np.array_equal(c32, c64) and np.array_equal(s32, s64)
    bad = w.copy()
    bad[rows - 2, 7] = np.inf
    with pytest.raises(ValueError):
        orc.quantize_f32(bad, fmt)
