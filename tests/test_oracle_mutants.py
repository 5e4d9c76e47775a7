"""The pins must be able to fail.  Each case below plants one plausible mistake
in a copy of the oracle's C source (a wrong exponent bias, a dropped term, a
swapped or transposed operand, a wrong index, a wrong tie-break or rounding
rule), builds that copy, and runs every pin of the oracle (the tests in
test_oracle_formats.py and test_oracle_route_layer.py) against it: at least
one pin has to fail.  The unmodified source, built and run through the same
harness, has to pass every pin, so a detection is not a harness error.

Everything here runs on the CPU.  The planted mistakes never index outside
the buffers the oracle allocates (each one was checked by reading), so a
mutant can give wrong numbers but cannot crash the test process."""
import contextlib
import ctypes
import importlib.util
import os
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "mx_oracle.c")

# (name, text in mx_oracle.c, replacement).  Each anchor occurs exactly once.
MUTANTS = [
    # element and scale decoding (OCP MX v1.0 formats)
    ("e4m3_bias_8", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("e4m3_subnormal_2^-7", "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    ("e4m3_nan_code_is_a_number", "if (e == 0xF && m == 7) return NAN;", ""),
    ("e2m1_bias_0", "ldexp(1.0 + (double)m / 2.0, e - 1)", "ldexp(1.0 + (double)m / 2.0, e)"),
    ("e2m1_subnormal_m", "double mag = (e == 0) ? (double)m / 2.0 :", "double mag = (e == 0) ? (double)m :"),
    ("e8m0_bias_128", "return ldexp(1.0, code - 127);", "return ldexp(1.0, code - 128);"),
    # block quantisation: shared exponent, rounding, saturation, signs
    ("floor_log2_off_by_one", "return x - 1;", "return x;"),
    ("e4m3_emax_7", "int emax = (fmt == ORC_E4M3) ? 8 : 2;", "int emax = (fmt == ORC_E4M3) ? 7 : 2;"),
    ("e2m1_emax_3", "int emax = (fmt == ORC_E4M3) ? 8 : 2;", "int emax = (fmt == ORC_E4M3) ? 8 : 3;"),
    ("amax_of_signed_values", "if (fabs(v[i]) > amax) amax = fabs(v[i]);", "if (v[i] > amax) amax = v[i];"),
    ("zero_block_scale_127", "int s = (amax == 0.0) ? -127 :", "int s = (amax == 0.0) ? 0 :"),
    ("no_lower_scale_clamp", "if (s < -127) s = -127;", ""),
    ("no_upper_scale_clamp", "if (s > 127) s = 127;", ""),
    ("nonfinite_accepted", "if (!isfinite(v[i])) return ORC_ERR_NONFINITE;", ""),
    ("e4m3_ties_away_from_zero", "double v = nearbyint(a / spacing) * spacing; /* a / spacing is exact; RNE */",
     "double v = round(a / spacing) * spacing;"),
    ("e4m3_truncates", "double v = nearbyint(a / spacing) * spacing; /* a / spacing is exact; RNE */",
     "double v = trunc(a / spacing) * spacing;"),
    ("e2m1_ties_away_from_zero", "double v = nearbyint(a / spacing) * spacing;\n  if (v > 6.0)",
     "double v = round(a / spacing) * spacing;\n  if (v > 6.0)"),
    ("e4m3_no_saturation", "if (v > 448.0) v = 448.0;", ""),
    ("e2m1_no_saturation", "if (v > 6.0) v = 6.0;", ""),
    ("e4m3_no_subnormal_binade", "int e = (a < ldexp(1.0, -6)) ? -6 : floor_log2(a);", "int e = floor_log2(a);"),
    ("negative_zero_loses_sign", "int sign = signbit(q) ? 0x80 : 0;", "int sign = (q < 0) ? 0x80 : 0;"),
    ("e2m1_packing_high_nibble_first", "if (col % 2 == 0) *p", "if (col % 2 == 1) *p"),
    # weight quantisation (fp32 rows, split over threads)
    ("f32_e2m1_row_stride_quarter", "int64_t row_bytes = (fmt == ORC_E4M3) ? K : K / 2;",
     "int64_t row_bytes = (fmt == ORC_E4M3) ? K : K / 4;"),
    ("f32_e4m3_row_stride_half", "int64_t row_bytes = (fmt == ORC_E4M3) ? K : K / 2;",
     "int64_t row_bytes = (fmt == ORC_E4M3) ? K / 2 : K / 2;"),
    ("f32_copies_row_0", "rowbuf[i] = (double)w[r * K + i];", "rowbuf[i] = (double)w[i];"),
    ("f32_scales_of_row_0", "codes + r * row_bytes, scales + r * (K / 32)", "codes + r * row_bytes, scales"),
    ("f32_status_dropped", "      if (rs) {\n#pragma omp atomic write\n        st = rs;\n      }\n", ""),
    # router
    ("topk_ties_to_highest_index", "(best < 0 || l[e] > l[best])", "(best < 0 || l[e] >= l[best])"),
    ("topk_ascending", "(best < 0 || l[e] > l[best])", "(best < 0 || l[e] < l[best])"),
    ("softmax_drops_last_term", "for (int j = 0; j < k; ++j) den += exp(",
     "for (int j = 0; j < k - 1; ++j) den += exp("),
    # permutation
    ("shared_count_zero", "counts[E] = T;", "counts[E] = 0;"),
    ("shared_slot_j_0", "sorted_slot[pos++] = t * (k + 1) + k;", "sorted_slot[pos++] = t * (k + 1);"),
    ("slot_id_stride_k", "sorted_slot[pos++] = t * (k + 1) + j;", "sorted_slot[pos++] = t * k + j;"),
    ("slots_ordered_by_position_first",
     "    for (int t = 0; t < T; ++t)\n      for (int j = 0; j < k; ++j)\n        if (ids",
     "    for (int j = 0; j < k; ++j)\n      for (int t = 0; t < T; ++t)\n        if (ids"),
    # expert layer
    ("weight_scale_of_row_0", "double s = orc_decode_e8m0(scales[r * (K / 32) + c / 32]);",
     "double s = orc_decode_e8m0(scales[c / 32]);"),
    ("e2m1_decode_high_nibble_first", "v = orc_decode_e2m1((c % 2 == 0) ?", "v = orc_decode_e2m1((c % 2 == 1) ?"),
    ("activation_scale_of_block_0", "orc_decode_e8m0(act_scales[(int64_t)t * (H / 32) + h / 32])",
     "orc_decode_e8m0(act_scales[(int64_t)t * (H / 32)])"),
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("gate_and_up_swapped", "hv[i] = silu(g) * u;", "hv[i] = silu(u) * g;"),
    ("up_from_gate_rows", "u += x[h] * w1d[(int64_t)(I + i) * H + h];", "u += x[h] * w1d[(int64_t)i * H + h];"),
    ("gate_weight_transposed", "g += x[h] * w1d[(int64_t)i * H + h];", "g += x[h] * w1d[(int64_t)h * I + i];"),
    ("down_weight_transposed", "y += hq[i] * w2d[(int64_t)o * I + i];", "y += hq[i] * w2d[(int64_t)i * H + o];"),
    ("h_not_requantised", "y += hq[i] * w2d", "y += hv[i] * w2d"),
    ("h_requantised_in_weight_format", "orc_quantize_rows(hv, 1, I, h_fmt, hc, hs)",
     "orc_quantize_rows(hv, 1, I, fmt, hc, hs)"),
    # SwiGLU-OAI and the MXFP4-activation variant
    ("oai_gate_clamped_below_too", "  if (g > limit) g = limit;\n", "  if (g > limit) g = limit;\n  if (g < -limit) g = -limit;\n"),
    ("oai_up_not_clamped", "  if (u > limit) u = limit;\n  if (u < -limit) u = -limit;\n", ""),
    ("oai_no_plus_one", "return g / (1.0 + exp(-alpha * g)) * (u + 1.0);", "return g / (1.0 + exp(-alpha * g)) * u;"),
    ("oai_alpha_outside_sigmoid", "return g / (1.0 + exp(-alpha * g)) * (u + 1.0);",
     "return alpha * g / (1.0 + exp(-g)) * (u + 1.0);"),
    ("fp4_act_high_nibble_first", "xv = orc_decode_e2m1((h % 2 == 0) ? (byte & 0xF) : (byte >> 4));",
     "xv = orc_decode_e2m1((h % 2 == 1) ? (byte & 0xF) : (byte >> 4));"),
    ("fp4_h_decoded_as_e4m3", "double hcv = (h_fmt == ORC_E4M3) ?", "double hcv = 1 ?"),
    # router GEMM and biased top-k
    ("router_weight_transposed", "bf16_to_double(w[(int64_t)e * H + h])", "bf16_to_double(w[(int64_t)h * E + e])"),
    ("router_drops_last_column", "      for (int h = 0; h < H; ++h)\n        acc +=", "      for (int h = 0; h < H - 1; ++h)\n        acc +="),
    ("biased_weights_from_scores", "den += exp((double)l[ids[(int64_t)t * k + jj]] - lmax);\n    for (int jj = 0; jj < k; ++jj) w[(int64_t)t * k + jj] = exp((double)l[ids[(int64_t)t * k + jj]] - lmax) / den;",
     "den += exp((double)score[ids[(int64_t)t * k + jj]] - lmax);\n    for (int jj = 0; jj < k; ++jj) w[(int64_t)t * k + jj] = exp((double)score[ids[(int64_t)t * k + jj]] - lmax) / den;"),
    ("biased_ties_to_highest", "if (!taken[e] && (best < 0 || score[e] > score[best])) best = e;",
     "if (!taken[e] && (best < 0 || score[e] >= score[best])) best = e;"),
    ("router_weight_dropped", "double wt = (j == k) ? 1.0 : topk_w[(int64_t)t * k + j];", "double wt = 1.0;"),
    ("shared_takes_first_router_weight", "double wt = (j == k) ? 1.0 : topk_w[(int64_t)t * k + j];",
     "double wt = (j == k) ? topk_w[(int64_t)t * k] : topk_w[(int64_t)t * k + j];"),
    ("shared_expert_left_out", "for (int e = 0; e <= E; ++e) {\n    /* the requested tokens",
     "for (int e = 0; e < E; ++e) {\n    /* the requested tokens"),
]


def _load_module(fname):
    spec = importlib.util.spec_from_file_location("_pins_" + fname, os.path.join(HERE, fname + ".py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _pin_calls():
    """Every pin, expanded over its parametrisation, in file order."""
    calls = []
    for mod in (_load_module("test_oracle_formats"), _load_module("test_oracle_route_layer")):
        for name, fn in vars(mod).items():
            if not name.startswith("test_") or not callable(fn):
                continue
            marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
            if not marks:
                calls.append((name, fn, {}))
                continue
            argnames, values = marks[0].args[0], marks[0].args[1]
            argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
            for v in values:
                v = tuple(v) if len(argnames) > 1 else (v,)
                calls.append((f"{name}{list(v)}", fn, dict(zip(argnames, v))))
    return calls


@contextlib.contextmanager
def _oracle_from(path):
    """Point the oracle's wrappers at another build of the C source."""
    saved_lib, saved_tables = oracle._lib, dict(oracle._tables)
    oracle._lib = oracle._bind(ctypes.CDLL(path))
    oracle._tables.clear()
    try:
        yield oracle
    finally:
        oracle.set_threads(0)
        oracle._lib = saved_lib
        oracle._tables.clear()
        oracle._tables.update(saved_tables)


def _failing_pins(orc, calls, stop_at_first):
    failed = []
    for name, fn, kw in calls:
        try:
            fn(orc, **kw)
        except (Exception, pytest.fail.Exception) as ex:  # an assertion, pytest.raises, or an oracle error status
            failed.append((name, type(ex).__name__))
            if stop_at_first:
                break
    return failed


@pytest.fixture(scope="module")
def builds(tmp_path_factory):
    """The unmodified source and every mutant, compiled in parallel."""
    with open(SRC) as f:
        text = f.read()
    d = tmp_path_factory.mktemp("oracle_mutants")
    jobs = {"unmodified": text}
    for name, old, new in MUTANTS:
        assert text.count(old) == 1, f"mutant {name}: anchor not found exactly once in mx_oracle.c"
        jobs[name] = text.replace(old, new)

    def one(item):
        name, src = item
        c = os.path.join(d, name + ".c")
        with open(c, "w") as f:
            f.write(src)
        return name, oracle.compile_library(c, os.path.join(d, "lib" + name + ".so"))

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        return dict(ex.map(one, jobs.items()))


@pytest.fixture(scope="module")
def pins():
    return _pin_calls()


def test_mutant_names_are_distinct():
    names = [m[0] for m in MUTANTS]
    assert len(names) == len(set(names))


def test_unmodified_copy_passes_every_pin(builds, pins):
    assert len(pins) > 20
    with _oracle_from(builds["unmodified"]) as orc:
        assert _failing_pins(orc, pins, stop_at_first=False) == []


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(builds, pins, name):
    with _oracle_from(builds[name]) as orc:
        failed = _failing_pins(orc, pins, stop_at_first=True)
    assert failed, f"no pin detects the planted mistake {name}"
