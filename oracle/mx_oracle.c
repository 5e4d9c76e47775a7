/*
 * mx_oracle.c -- plain, slow, CPU reference ("oracle") for the MX block-scaled
 * sparse-MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library and follows the method step by step, in double precision:
 *
 *   - MX element formats (E4M3, E2M1) and the E8M0 block scale, as fixed by the
 *     OCP Microscaling Formats (MX) v1.0 specification, the formats the pages
 *     name for MXFP8 / MXFP4 weights ("Tracing the bottleneck: optimising
 *     MiniMax M3 on AMD Instinct MI355X", opening results list and Figure 1).
 *   - Block quantisation: shared exponent = floor(log2(amax)) - emax(element),
 *     elements divided by 2^exponent, rounded to nearest even, saturated.
 *   - Router: top-k of fp32 logits with lowest-index tie-break, softmax over
 *     the k selected logits.
 *   - The shared expert folded into the routed table as an always-selected
 *     expert with weight 1 (same page, Figure 4).
 *   - Token -> expert permutation: experts ascending (shared last), tokens
 *     ascending inside an expert.
 *   - Expert MLP: g = x.Wg, u = x.Wu, h = silu(g) * u (or the SwiGLU-OAI form
 *     with a clamp limit and a sigmoid slope, same page, correctness passage),
 *     h re-quantised per 32 along I to MXFP8 (MXFP4 when the activations are
 *     MXFP4: the page's MXFP4 results), y = h.Wd, out[t] += w * y  (the down projection with the
 *     weighted combine, "Kimi K3 performance in vLLM: 2.8x throughput",
 *     section on fusing the MXFP4 top-k finalize into the epilogue).
 *
 * All sums are plain fp64 loops in index order; no blocking or reordering.
 * Non-finite inputs are a precondition violation and return ORC_ERR_NONFINITE.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_NONFINITE 2
#define ORC_ERR_NOMEM 3

#define ORC_E4M3 0
#define ORC_E2M1 1

/* ------------------------------------------------------------------ decode */

/* E4M3 (OCP MX v1.0): sign, 4 exponent bits (bias 7), 3 mantissa bits.
 * e == 0 is subnormal: 2^-6 * m/8.  S.1111.111 is NaN; there is no infinity. */
double orc_decode_e4m3(int code) {
  code &= 0xFF;
  int s = code >> 7, e = (code >> 3) & 0xF, m = code & 7;
  if (e == 0xF && m == 7) return NAN;
  double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* E2M1 (OCP MX v1.0): sign, 2 exponent bits (bias 1), 1 mantissa bit.
 * e == 0 is subnormal: 2^0 * m/2.  No infinity, no NaN.  Uses the low nibble. */
double orc_decode_e2m1(int code) {
  code &= 0xF;
  int s = code >> 3, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? (double)m / 2.0 : ldexp(1.0 + (double)m / 2.0, e - 1);
  return s ? -mag : mag;
}

/* E8M0 scale (OCP MX v1.0): 2^(code - 127); 0xFF is NaN. */
double orc_decode_e8m0(int code) {
  code &= 0xFF;
  if (code == 0xFF) return NAN;
  return ldexp(1.0, code - 127);
}

/* ------------------------------------------------------------------ encode */

/* Largest e with 2^e <= a, for finite a > 0 (exact: frexp gives a = f*2^x,
 * f in [0.5, 1)). */
static int floor_log2(double a) {
  int x;
  frexp(a, &x);
  return x - 1;
}

/* Round |q| to the nearest E4M3 magnitude, ties to even, saturating at 448;
 * return the code with the sign of q kept (so -tiny encodes as -0, 0x80). */
static int encode_e4m3(double q) {
  int sign = signbit(q) ? 0x80 : 0;
  double a = fabs(q);
  /* grid spacing in the binade of a; all subnormals share the spacing 2^-9 */
  int e = (a < ldexp(1.0, -6)) ? -6 : floor_log2(a);
  double spacing = ldexp(1.0, e - 3);
  double v = nearbyint(a / spacing) * spacing; /* a / spacing is exact; RNE */
  if (v > 448.0) v = 448.0;
  int code;
  if (v < ldexp(1.0, -6)) {
    code = (int)(v / ldexp(1.0, -9)); /* subnormal: v = m * 2^-9 */
  } else {
    int ev = floor_log2(v);
    int m = (int)((ldexp(v, -ev) - 1.0) * 8.0);
    code = ((ev + 7) << 3) | m;
  }
  return sign | code;
}

/* Round |q| to the nearest E2M1 magnitude, ties to even, saturating at 6. */
static int encode_e2m1(double q) {
  int sign = signbit(q) ? 0x8 : 0;
  double a = fabs(q);
  int e = (a < 1.0) ? 0 : floor_log2(a);
  double spacing = ldexp(1.0, e - 1);
  double v = nearbyint(a / spacing) * spacing;
  if (v > 6.0) v = 6.0;
  int code;
  if (v < 1.0) {
    code = (int)(v / 0.5);
  } else {
    int ev = floor_log2(v);
    int m = (int)((ldexp(v, -ev) - 1.0) * 2.0);
    code = ((ev + 1) << 1) | m;
  }
  return sign | code;
}

/* Quantise one block of n values to `fmt`.  codes[] gets one (unpacked) code
 * per element.  Shared exponent s = floor(log2(amax)) - emax, emax = 8 for
 * E4M3 and 2 for E2M1, clamped to the E8M0 range [-127, 127]; an all-zero block
 * has log2(0) = -inf and so takes the clamp, scale code 0. */
int orc_quantize_block(const double* v, int n, int fmt, uint8_t* codes, uint8_t* scale_code) {
  if (!v || !codes || !scale_code || n <= 0 || (fmt != ORC_E4M3 && fmt != ORC_E2M1)) return ORC_ERR_ARG;
  double amax = 0.0;
  for (int i = 0; i < n; ++i) {
    if (!isfinite(v[i])) return ORC_ERR_NONFINITE;
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  }
  int emax = (fmt == ORC_E4M3) ? 8 : 2;
  int s = (amax == 0.0) ? -127 : floor_log2(amax) - emax;
  if (s < -127) s = -127;
  if (s > 127) s = 127;
  *scale_code = (uint8_t)(s + 127);
  for (int i = 0; i < n; ++i) {
    double q = ldexp(v[i], -s); /* exact: division by a power of two */
    codes[i] = (uint8_t)(fmt == ORC_E4M3 ? encode_e4m3(q) : encode_e2m1(q));
  }
  return ORC_OK;
}

/* Quantise a [rows, K] matrix, blocks of 32 along K.  E4M3 codes are one byte
 * per element; E2M1 codes are packed two per byte, element 2i in the low
 * nibble.  scales: [rows, K/32]. */
int orc_quantize_rows(const double* v, int64_t rows, int64_t K, int fmt, uint8_t* codes,
                      uint8_t* scales) {
  if (!v || !codes || !scales || rows < 0 || K <= 0 || K % 32) return ORC_ERR_ARG;
  uint8_t blk[32];
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < K / 32; ++b) {
      int st = orc_quantize_block(v + r * K + b * 32, 32, fmt, blk, scales + r * (K / 32) + b);
      if (st) return st;
      for (int i = 0; i < 32; ++i) {
        int64_t col = b * 32 + i;
        if (fmt == ORC_E4M3) {
          codes[r * K + col] = blk[i];
        } else {
          uint8_t* p = codes + r * (K / 2) + col / 2;
          if (col % 2 == 0) *p = (uint8_t)((*p & 0xF0) | (blk[i] & 0xF));
          else *p = (uint8_t)((*p & 0x0F) | ((blk[i] & 0xF) << 4));
        }
      }
    }
  }
  return ORC_OK;
}

static double bf16_to_double(uint16_t b) {
  union { uint32_t u; float f; } c;
  c.u = (uint32_t)b << 16;
  return (double)c.f;
}

/* Activation quantisation: bf16 [rows, K] -> MXFP8 (E4M3 codes + E8M0). */
int orc_quantize_bf16(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales) {
  if (!x || rows < 0 || K <= 0 || K % 32) return ORC_ERR_ARG;
  double* row = (double*)malloc(sizeof(double) * (size_t)K);
  if (!row) return ORC_ERR_NOMEM;
  int st = ORC_OK;
  for (int64_t r = 0; r < rows && st == ORC_OK; ++r) {
    for (int64_t i = 0; i < K; ++i) row[i] = bf16_to_double(x[r * K + i]);
    st = orc_quantize_rows(row, 1, K, ORC_E4M3, codes + r * K, scales + r * (K / 32));
  }
  free(row);
  return st;
}

/* Weight quantisation: fp32 [rows, K] -> MXFP8 or MXFP4. */
int orc_quantize_f32(const float* w, int64_t rows, int64_t K, int fmt, uint8_t* codes,
                     uint8_t* scales) {
  if (!w || !codes || !scales || rows < 0 || K <= 0 || K % 32) return ORC_ERR_ARG;
  if (fmt != ORC_E4M3 && fmt != ORC_E2M1) return ORC_ERR_ARG;
  int64_t row_bytes = (fmt == ORC_E4M3) ? K : K / 2;
  int st = ORC_OK;
  /* rows are independent: one row per iteration */
#pragma omp parallel
  {
    double* rowbuf = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      if (!rowbuf) continue;
      for (int64_t i = 0; i < K; ++i) rowbuf[i] = (double)w[r * K + i];
      int rs = orc_quantize_rows(rowbuf, 1, K, fmt, codes + r * row_bytes, scales + r * (K / 32));
      if (rs) {
#pragma omp atomic write
        st = rs;
      }
    }
    if (!rowbuf) {
#pragma omp atomic write
      st = ORC_ERR_NOMEM;
    }
    free(rowbuf);
  }
  return st;
}

/* ------------------------------------------------------------------ router */

/* Top-k of each token's E logits: repeatedly take the largest remaining logit,
 * the lowest expert index winning ties, so ids come out in descending logit
 * order.  w = softmax over the k selected logits, in fp64. */
int orc_route_topk(const float* logits, int T, int E, int k, int32_t* ids, double* w) {
  if (!logits || !ids || !w || T < 0 || E <= 0 || k <= 0 || k > E) return ORC_ERR_ARG;
  char* taken = (char*)malloc((size_t)E);
  if (!taken) return ORC_ERR_NOMEM;
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    for (int e = 0; e < E; ++e) {
      if (!isfinite(l[e])) { free(taken); return ORC_ERR_NONFINITE; }
      taken[e] = 0;
    }
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
      taken[best] = 1;
      ids[(int64_t)t * k + j] = best;
    }
    double lmax = (double)l[ids[(int64_t)t * k]];
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += exp((double)l[ids[(int64_t)t * k + j]] - lmax);
    for (int j = 0; j < k; ++j)
      w[(int64_t)t * k + j] = exp((double)l[ids[(int64_t)t * k + j]] - lmax) / den;
  }
  free(taken);
  return ORC_OK;
}

/* Router GEMM (the step ahead of top-k): logits[t, e] = sum_h x[t, h] * w[e, h]
 * for bf16 activations x [T, H] and bf16 router weights w [E, H], products and
 * sums in fp64 (each bf16 product is exact in fp64).  The pages route tokens
 * to experts by their router logits (the MI355X page, Figure 4 and the
 * passage around it) without printing the router; a linear map of the hidden
 * state is the plain reading. */
int orc_router_logits(const uint16_t* x, const uint16_t* w, int T, int H, int E, double* logits) {
  if (!x || !w || !logits || T < 0 || H <= 0 || E <= 0) return ORC_ERR_ARG;
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += bf16_to_double(x[(int64_t)t * H + h]) * bf16_to_double(w[(int64_t)e * H + h]);
      logits[(int64_t)t * E + e] = acc;
    }
  return ORC_OK;
}

/* Top-k with a load-balancing bias: experts are chosen by the fp32 score
 * logit + bias[e] (the addition done in fp32, as the selection runs on the
 * GPU), largest first, lowest index on ties; the weights are the softmax of
 * the chosen experts' unbiased logits (fp64).  Reading: the bias steers which
 * experts are chosen, not how much each contributes.  bias = NULL is
 * orc_route_topk. */
int orc_route_topk_biased(const float* logits, const float* bias, int T, int E, int k, int32_t* ids, double* w) {
  if (!logits || !ids || !w || T < 0 || E <= 0 || k <= 0 || k > E) return ORC_ERR_ARG;
  float* score = (float*)malloc(sizeof(float) * (size_t)E);
  char* taken = (char*)malloc((size_t)E);
  if (!score || !taken) { free(score); free(taken); return ORC_ERR_NOMEM; }
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    for (int e = 0; e < E; ++e) {
      if (!isfinite(l[e]) || (bias && !isfinite(bias[e]))) { free(score); free(taken); return ORC_ERR_NONFINITE; }
      volatile float sum = l[e] + (bias ? bias[e] : 0.0f); /* one fp32 addition */
      score[e] = sum;
      taken[e] = 0;
    }
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || score[e] > score[best])) best = e;
      taken[best] = 1;
      ids[(int64_t)t * k + j] = best;
    }
    double lmax = -INFINITY;
    for (int j = 0; j < k; ++j) {
      double v = (double)l[ids[(int64_t)t * k + j]];
      if (v > lmax) lmax = v;
    }
    double den = 0.0;
    for (int jj = 0; jj < k; ++jj) den += exp((double)l[ids[(int64_t)t * k + jj]] - lmax);
    for (int jj = 0; jj < k; ++jj) w[(int64_t)t * k + jj] = exp((double)l[ids[(int64_t)t * k + jj]] - lmax) / den;
  }
  free(score);
  free(taken);
  return ORC_OK;
}

/* ------------------------------------------------------------------ permute */

/* counts[e] = tokens routed to expert e (e < E), counts[E] = T (the shared
 * expert takes every token); offsets = exclusive prefix of counts, E + 2
 * entries; sorted_slot lists slot ids t*(k+1)+j grouped by expert ascending
 * (shared last), tokens ascending inside each expert.  j = k is the shared
 * slot. */
int orc_permute(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                int32_t* sorted_slot) {
  if (!ids || !counts || !offsets || !sorted_slot || T < 0 || E <= 0 || k <= 0) return ORC_ERR_ARG;
  for (int e = 0; e <= E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < (int64_t)T * k; ++i) {
    if (ids[i] < 0 || ids[i] >= E) return ORC_ERR_ARG;
    counts[ids[i]]++;
  }
  counts[E] = T;
  offsets[0] = 0;
  for (int e = 0; e <= E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int64_t pos = 0;
  for (int e = 0; e < E; ++e)
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (ids[(int64_t)t * k + j] == e) sorted_slot[pos++] = t * (k + 1) + j;
  for (int t = 0; t < T; ++t) sorted_slot[pos++] = t * (k + 1) + k;
  return ORC_OK;
}

/* ------------------------------------------------------------------ expert layer */

static double silu(double z) { return z / (1.0 + exp(-z)); }

#define ORC_ACT_SWIGLU 0
#define ORC_ACT_SWIGLU_OAI 1

/* SwiGLU-OAI ("Tracing the bottleneck: optimising MiniMax M3 on AMD Instinct
 * MI355X", correctness passage: the model's SwiGLU-OAI parameters are passed
 * into the MoE; the page gives neither the formula nor the values).  Reading:
 * the gate is clamped above at `limit`, the up projection to [-limit, limit],
 * h = g * sigmoid(alpha * g) * (u + 1).  Parity unpinned beyond the special
 * cases the tests reduce to textbook functions (limit = 0; alpha = 1 with no
 * clamp). */
double orc_swiglu_oai(double g, double u, double alpha, double limit) {
  if (g > limit) g = limit;
  if (u > limit) u = limit;
  if (u < -limit) u = -limit;
  return g / (1.0 + exp(-alpha * g)) * (u + 1.0);
}

/* Decode an MX matrix [rows, K] (codes in `fmt`, E8M0 scales per 32) to fp64. */
static void decode_matrix(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t K,
                          int fmt, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < K; ++c) {
      double s = orc_decode_e8m0(scales[r * (K / 32) + c / 32]);
      double v;
      if (fmt == ORC_E4M3) {
        v = orc_decode_e4m3(codes[r * K + c]);
      } else {
        uint8_t byte = codes[r * (K / 2) + c / 2];
        v = orc_decode_e2m1((c % 2 == 0) ? (byte & 0xF) : (byte >> 4));
      }
      out[r * K + c] = v * s;
    }
}

/*
 * The expert layer on already-quantised activations.
 *   act_codes/act_scales: MX activations in `act_fmt` ([T, H] E4M3 codes or
 *     [T, H/2] packed E2M1 codes), scales [T, H/32].
 *   ids/topk_w: router output [T, k].
 *   w1c/w1s[e], w2c/w2s[e], e = 0..E (E = shared): canonical MX weights,
 *     W1 [2I, H] (rows 0..I-1 gate, I..2I-1 up), W2 [H, I]; a NULL entry is
 *     allowed for an expert none of the requested tokens uses.
 *   tokens[n_tokens]: distinct token indices to evaluate (NULL = all T).
 *   out[n_tokens, H]: fp64 result, rows in the order of `tokens`.
 *   out_noq (optional): the same layer with h left unquantised.
 *   h_codes/h_scales (optional): h per slot id t*(k+1)+j in `h_fmt`,
 *     [T*(k+1), I] (E4M3) or [T*(k+1), I/2] (E2M1) and [T*(k+1), I/32]; rows of
 *     tokens not requested are left untouched.
 *   act: ORC_ACT_SWIGLU (h = silu(g) * u) or ORC_ACT_SWIGLU_OAI with `alpha`
 *     and `limit` (orc_swiglu_oai).
 *   h_fmt: the MX element format h is re-quantised to (E4M3; E2M1 for the
 *     variant with MXFP4 activations, whose both MMA operands are E2M1).
 * Experts are visited in ascending order (shared last) and each token's
 * contributions are added in that order.
 */
int orc_expert_layer_ex(const uint8_t* act_codes, const uint8_t* act_scales, int T, int H, int I,
                        int E, int k, const int32_t* ids, const double* topk_w,
                        const uint8_t* const* w1c, const uint8_t* const* w1s,
                        const uint8_t* const* w2c, const uint8_t* const* w2s, int fmt,
                        const int32_t* tokens, int n_tokens, double* out, double* out_noq,
                        uint8_t* h_codes, uint8_t* h_scales, int act, double alpha, double limit,
                        int act_fmt, int h_fmt) {
  if (!act_codes || !act_scales || !ids || !topk_w || !w1c || !w1s || !w2c || !w2s || !out)
    return ORC_ERR_ARG;
  if (T < 0 || H <= 0 || I <= 0 || H % 32 || I % 32 || E <= 0 || k <= 0 || k > E) return ORC_ERR_ARG;
  if (fmt != ORC_E4M3 && fmt != ORC_E2M1) return ORC_ERR_ARG;
  if (act != ORC_ACT_SWIGLU && act != ORC_ACT_SWIGLU_OAI) return ORC_ERR_ARG;
  if ((act_fmt != ORC_E4M3 && act_fmt != ORC_E2M1) || (h_fmt != ORC_E4M3 && h_fmt != ORC_E2M1)) return ORC_ERR_ARG;
  /* row bytes of the activation and h codes: one byte per element (E4M3) or
   * two elements per byte, element 2i in the low nibble (E2M1) */
  const int64_t act_row = (act_fmt == ORC_E4M3) ? H : H / 2;
  const int64_t h_row = (h_fmt == ORC_E4M3) ? I : I / 2;
  if (!tokens) n_tokens = T;
  int* row_of = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
  double* xd = (double*)malloc(sizeof(double) * (size_t)n_tokens * H + 1);
  double* w1d = (double*)malloc(sizeof(double) * (size_t)2 * I * H);
  double* w2d = (double*)malloc(sizeof(double) * (size_t)H * I);
  int* slot_tok = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
  int* slot_j = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
  double* ybuf = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * H);
  double* ybuf_noq = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * H);
  int st = ORC_OK;
  if (!row_of || !xd || !w1d || !w2d || !slot_tok || !slot_j || !ybuf || !ybuf_noq) {
    st = ORC_ERR_NOMEM;
    goto done;
  }
  for (int t = 0; t < T; ++t) row_of[t] = -1;
  for (int r = 0; r < n_tokens; ++r) {
    int t = tokens ? tokens[r] : r;
    if (t < 0 || t >= T || row_of[t] >= 0) { st = ORC_ERR_ARG; goto done; }
    row_of[t] = r;
  }
  for (int r = 0; r < n_tokens; ++r) {
    int t = tokens ? tokens[r] : r;
    for (int h = 0; h < H; ++h) {
      double xv;
      if (act_fmt == ORC_E4M3) {
        xv = orc_decode_e4m3(act_codes[(int64_t)t * H + h]);
      } else {
        uint8_t byte = act_codes[(int64_t)t * act_row + h / 2];
        xv = orc_decode_e2m1((h % 2 == 0) ? (byte & 0xF) : (byte >> 4));
      }
      xd[(int64_t)r * H + h] = xv * orc_decode_e8m0(act_scales[(int64_t)t * (H / 32) + h / 32]);
    }
  }
  for (int64_t i = 0; i < (int64_t)n_tokens * H; ++i) out[i] = 0.0;
  if (out_noq)
    for (int64_t i = 0; i < (int64_t)n_tokens * H; ++i) out_noq[i] = 0.0;

  for (int e = 0; e <= E; ++e) {
    /* the requested tokens routed to e, ascending, with their top-k position */
    int ns = 0;
    for (int t = 0; t < T; ++t) {
      if (row_of[t] < 0) continue;
      int jj = -1;
      if (e == E) jj = k;
      else
        for (int j = 0; j < k; ++j)
          if (ids[(int64_t)t * k + j] == e) jj = j;
      if (jj < 0) continue;
      slot_tok[ns] = t;
      slot_j[ns] = jj;
      ns++;
    }
    if (ns == 0) continue;
    if (!w1c[e] || !w1s[e] || !w2c[e] || !w2s[e]) { st = ORC_ERR_ARG; goto done; }
    decode_matrix(w1c[e], w1s[e], 2 * (int64_t)I, H, fmt, w1d);
    decode_matrix(w2c[e], w2s[e], H, I, fmt, w2d);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int si = 0; si < ns; ++si) {
      int t = slot_tok[si];
      const double* x = xd + (int64_t)row_of[t] * H;
      double* hv = (double*)malloc(sizeof(double) * (size_t)I * 2);
      uint8_t* hc = (uint8_t*)malloc((size_t)I + (size_t)I / 32);
      if (!hv || !hc) {
        free(hv); free(hc);
#pragma omp atomic write
        bad = ORC_ERR_NOMEM;
        continue;
      }
      double* hq = hv + I;
      for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
          g += x[h] * w1d[(int64_t)i * H + h];
          u += x[h] * w1d[(int64_t)(I + i) * H + h];
        }
        if (act == ORC_ACT_SWIGLU_OAI) hv[i] = orc_swiglu_oai(g, u, alpha, limit);
        else hv[i] = silu(g) * u;
      }
      /* re-quantise h per 32 along I (MXFP8, or MXFP4 with FP4 activations) */
      uint8_t* hs = hc + I;
      int qst = orc_quantize_rows(hv, 1, I, h_fmt, hc, hs);
      if (qst) {
#pragma omp atomic write
        bad = qst;
      }
      for (int i = 0; i < I; ++i) {
        double hcv = (h_fmt == ORC_E4M3) ? orc_decode_e4m3(hc[i])
                                          : orc_decode_e2m1((i % 2 == 0) ? (hc[i / 2] & 0xF) : (hc[i / 2] >> 4));
        hq[i] = hcv * orc_decode_e8m0(hs[i / 32]);
      }
      if (h_codes && h_scales) {
        int64_t sid = (int64_t)t * (k + 1) + slot_j[si];
        memcpy(h_codes + sid * h_row, hc, (size_t)h_row);
        memcpy(h_scales + sid * (I / 32), hs, (size_t)I / 32);
      }
      for (int o = 0; o < H; ++o) {
        double y = 0.0, y2 = 0.0;
        for (int i = 0; i < I; ++i) {
          y += hq[i] * w2d[(int64_t)o * I + i];
          y2 += hv[i] * w2d[(int64_t)o * I + i];
        }
        ybuf[(int64_t)si * H + o] = y;
        ybuf_noq[(int64_t)si * H + o] = y2;
      }
      free(hv);
      free(hc);
    }
    if (bad) { st = bad; goto done; }
    /* weighted combine, in slot order (token ascending) */
    for (int si = 0; si < ns; ++si) {
      int t = slot_tok[si], j = slot_j[si];
      double wt = (j == k) ? 1.0 : topk_w[(int64_t)t * k + j];
      double* o = out + (int64_t)row_of[t] * H;
      for (int h = 0; h < H; ++h) o[h] += wt * ybuf[(int64_t)si * H + h];
      if (out_noq) {
        double* o2 = out_noq + (int64_t)row_of[t] * H;
        for (int h = 0; h < H; ++h) o2[h] += wt * ybuf_noq[(int64_t)si * H + h];
      }
    }
  }
done:
  free(row_of); free(xd); free(w1d); free(w2d); free(slot_tok); free(slot_j); free(ybuf); free(ybuf_noq);
  return st;
}

/* The expert layer with the defaults: standard SwiGLU, MXFP8 activations and
 * MXFP8 h (see orc_expert_layer_ex). */
int orc_expert_layer(const uint8_t* act_codes, const uint8_t* act_scales, int T, int H, int I,
                     int E, int k, const int32_t* ids, const double* topk_w,
                     const uint8_t* const* w1c, const uint8_t* const* w1s,
                     const uint8_t* const* w2c, const uint8_t* const* w2s, int fmt,
                     const int32_t* tokens, int n_tokens, double* out, double* out_noq,
                     uint8_t* h_codes, uint8_t* h_scales) {
  return orc_expert_layer_ex(act_codes, act_scales, T, H, I, E, k, ids, topk_w, w1c, w1s, w2c, w2s, fmt,
                             tokens, n_tokens, out, out_noq, h_codes, h_scales, ORC_ACT_SWIGLU, 1.0,
                             INFINITY, ORC_E4M3, ORC_E4M3);
}

/* Number of OpenMP threads the oracle's parallel loops use from now on (the
   results do not depend on it: every output is computed by one thread in index
   order).  n <= 0 restores the runtime default. */
void orc_set_threads(int n) {
  if (n > 0) omp_set_num_threads(n);
  else omp_set_num_threads(omp_get_num_procs());
}
