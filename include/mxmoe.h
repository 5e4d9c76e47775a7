/*
 * mxmoe.h -- C ABI of libmxmoe.so, the GB300 (sm_103a) MX block-scaled
 * sparse-MoE expert layer.
 *
 * The layer (one MoE block of a transformer) computes, for T tokens of hidden
 * size H, E routed experts with intermediate size I and top-k routing, plus one
 * shared expert folded into the expert table at index E as an always-selected
 * expert of weight 1:
 *
 *   act      = MXFP8(x)                                   mx_quantize_act
 *   ids, w   = top-k(logits), softmax over the k chosen    moe_route_topk
 *   slots    = tokens grouped by expert                   moe_permute
 *   h[s]     = MXFP8( silu(act[t].Wg[e]) * (act[t].Wu[e]) ) moe_grouped_gemm_swiglu
 *   out[t]  += w[s] * (h[s] . Wd[e])                      moe_grouped_gemm_down_combine
 *
 * Sources: the MX weight formats and the shared-expert folding follow
 * "Tracing the bottleneck: optimising MiniMax M3 on AMD Instinct MI355X"
 * (opening results list for MXFP8/MXFP4 weights; Figure 4 for the shared
 * expert placed in the routed table and selected for every token; Figure 3 and
 * the surrounding passage for separate small-M / large-M schedules; the
 * passage after Figure 4 for moving weight/scale re-layout to load time).  The
 * combine fused into the down projection's epilogue follows "Kimi K3
 * performance in vLLM: 2.8x throughput" (section on fusing the MXFP4 top-k
 * finalize into the epilogue).  The element formats are those of the OCP
 * Microscaling Formats (MX) v1.0 specification.
 *
 * Conventions for every call
 *  - Pointers are DEVICE pointers owned by the caller unless stated; the
 *    library never allocates and never synchronises the stream.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous: they validate arguments on the host, enqueue kernels and
 *    return.  A return of MX_OK means the work was enqueued.
 *  - Device-side errors (a bounded wait that ran out, an expert id out of
 *    range) are OR-ed into a status word at the start of the caller's
 *    workspace; read and clear it with moe_get_status.
 *  - Workspaces must be zero-filled once before their first use (the library
 *    leaves them ready for the next call).
 *  - Formats: MX_E4M3 (MXFP8, one byte per element) and MX_E2M1 (MXFP4, two
 *    elements per byte, element 2i in the low nibble).  Every 32 consecutive
 *    elements along K share one E8M0 scale byte (value 2^(code-127)).
 *  - Non-finite inputs are a precondition violation: results are unspecified.
 */
#ifndef MXMOE_H_
#define MXMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mx_stream_t; /* same type as cudaStream_t */

#if defined(__GNUC__)
#define MX_API __attribute__((visibility("default")))
#else
#define MX_API
#endif

/* ---- status codes ---- */
#define MX_OK 0
#define MX_ERR_INVALID_ARG 1  /* null pointer, non-positive size, k > E, k > 32 ... */
#define MX_ERR_UNSUPPORTED 2  /* shape the kernels do not handle (see each call) */
#define MX_ERR_ALIGNMENT 3    /* a pointer is not 16-byte (weights: 256-byte) aligned */
#define MX_ERR_WORKSPACE 4    /* workspace / destination smaller than required */
#define MX_ERR_CUDA 5         /* a CUDA runtime/driver call or kernel launch failed */
#define MX_ERR_TIMEOUT 6      /* device status: a bounded wait inside a kernel ran out */
#define MX_ERR_DEVICE_ARG 7   /* device status: an expert id or slot id out of range */

/* ---- element formats ---- */
#define MX_E4M3 0
#define MX_E2M1 1

/* Human-readable name of a status code (static string, never NULL). */
MX_API const char* mx_status_string(int status);

/* Activation quantisation, bf16 -> MXFP8 (E4M3 codes + E8M0 scales).
 *   x_bf16  [T, H] row-major bf16.  codes [T, H] bytes.  scales [T, H/32] bytes.
 * Per row and per block of 32 along H: shared exponent
 * s = clamp(floor(log2(amax)) - 8, -127, 127) (an all-zero block gives -127),
 * scale byte s + 127, element code = E4M3 value of x / 2^s rounded to nearest
 * even and saturated to +-448; a negative value that rounds to zero keeps its
 * sign (0x80).  Bit-exact with the reference definition.
 * Errors: MX_ERR_INVALID_ARG (null, T < 0, H <= 0), MX_ERR_UNSUPPORTED
 * (H % 32), MX_ERR_ALIGNMENT (x or codes not 16-byte aligned).
 * Source: the MI355X page (opening results list: MXFP8 and MXFP4 models;
 * the passage on the native MXFP8 linear backend); the element and scale rule
 * is that of OCP MX v1.0. */
MX_API int mx_quantize_act(const void* x_bf16, int T, int H, uint8_t* codes, uint8_t* scales,
                    mx_stream_t stream);

/* mx_quantize_act to a chosen MX format: fmt MX_E4M3 (as mx_quantize_act) or
 * MX_E2M1 (MXFP4: emax 2, codes [T, H/2] bytes, element 2i in the low nibble,
 * saturation at 6), scales [T, H/32].  Errors as mx_quantize_act, plus
 * MX_ERR_INVALID_ARG for another fmt.  Source: as mx_quantize_act; MXFP4
 * activations are the mx_layer_opts act_fmt variant. */
MX_API int mx_quantize_act_ex(const void* x_bf16, int T, int H, int fmt, uint8_t* codes, uint8_t* scales,
                              mx_stream_t stream);

/* Weight quantisation, fp32 -> MXFP8 or MXFP4 (load-time helper; same rule as
 * mx_quantize_act with emax 8 for E4M3 and 2 for E2M1, saturation at 6 for
 * E2M1).  w [rows, K] fp32; codes [rows, K] (E4M3) or [rows, K/2] (E2M1);
 * scales [rows, K/32].  Errors as mx_quantize_act (K % 32). */
MX_API int mx_quantize_weights(const float* w, int64_t rows, int K, int fmt, uint8_t* codes,
                        uint8_t* scales, mx_stream_t stream);

/* Router: per token, the k largest of E fp32 logits, ties to the lowest expert
 * index, in descending logit order, and their softmax (over the k selected).
 *   logits [T, E] fp32; topk_ids [T, k] int32; topk_w [T, k] fp32.
 * Ids are bit-exact with the reference; weights are fp32 (a few ulp).
 * Errors: MX_ERR_INVALID_ARG (null, T < 0, E <= 0, k < 1, k > E, k > 32),
 * MX_ERR_UNSUPPORTED (E > 1024).
 * Source: the MI355X page, Figure 4 and its passage (each token's routed
 * experts, with the shared expert added as a slot every token selects) and the
 * correctness passage (the expert mask a token is routed through must be
 * exact); the Kimi K3 page, section on the MXFP4 top-k finalize.  The pages fix
 * no tie rule: lowest index first is this library's reading. */
MX_API int moe_route_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                   mx_stream_t stream);

/* Router GEMM with top-k in its epilogue (the step ahead of moe_route_topk):
 *   logits[t, e] = sum_h x[t, h] * w_router[e, h]   (bf16 inputs, fp32 accumulation;
 *     products of bf16 values are exact in fp32)
 *   topk_ids[t, :] = the k experts with the largest score logit + bias[e]
 *     (one fp32 addition), lowest index on ties, descending score order
 *   topk_w[t, :] = softmax of the chosen experts' unbiased logits (fp32).
 *   x_bf16 [T, H], w_router_bf16 [E, H] row-major, 16-byte aligned.
 *   bias [E] fp32 or NULL (no bias): a load-balancing bias that steers which
 *     experts are chosen but not their weights (this library's reading; the
 *     pages give no router).  logits [T, E] or NULL.  topk_ids and topk_w
 *     both NULL: logits only (then logits must be given).
 *   ws: a 256-byte-aligned workspace of at least 256 bytes, zero-filled once;
 *     its first word is the status word moe_get_status reads, its second a
 *     counter of the small-batch kernel.
 * Up to 128 tokens with somewhere to keep the logits (logits given, or ws of
 * at least 256 + 4*T*E bytes) run a CUDA-core kernel over blocks of 2 experts
 * (the router is then a weight-streaming matrix-vector product) whose last
 * block selects; larger batches run the tensor-core GEMM with the selection
 * in its epilogue.  Both sum the same exact bf16 products in fp32 (in
 * different orders).
 * Errors: MX_ERR_INVALID_ARG, MX_ERR_UNSUPPORTED (H % 64, E > 512, k > 16),
 * MX_ERR_ALIGNMENT, MX_ERR_WORKSPACE.
 * Source: the MI355X page, Figure 4 and its passage (tokens are routed to
 * experts by router scores; the router itself is not printed). */
MX_API int moe_route_gemm_topk(const void* x_bf16, const void* w_router_bf16, const float* bias, int T, int H,
                               int E, int k, float* logits, int32_t* topk_ids, float* topk_w, void* ws,
                               size_t ws_bytes, mx_stream_t stream);

/* Bytes of workspace moe_permute needs. */
MX_API size_t moe_permute_workspace_size(int T, int E, int k);

/* Token -> expert permutation with the shared expert folded in.
 *   counts [E+1]: tokens per expert, counts[E] = T (shared expert).
 *   offsets [E+2]: exclusive prefix of counts, offsets[E+1] = T*(k+1).
 *   sorted_slot [T*(k+1)]: slot ids t*(k+1)+j (j = k is the shared slot),
 *     grouped by expert ascending (shared last), tokens ascending inside each
 *     expert.  Bit-exact, deterministic, no host synchronisation.
 * topk_ids must hold k distinct ids in [0, E) per token; an id out of range
 * sets MX_ERR_DEVICE_ARG in the workspace status and is skipped.
 * Errors: MX_ERR_INVALID_ARG, MX_ERR_UNSUPPORTED (E > 1024),
 * MX_ERR_WORKSPACE (ws_bytes < moe_permute_workspace_size).
 * Source: the MI355X page, Figure 3 and its passage (the routed token count of
 * each expert is that expert's local M; grouped MoE programs are ordered so
 * that neighbours reuse activation rows and expert weight tiles) and Figure 4
 * (the shared expert sits in the routed table and the grouped GEMMs process it
 * in the same pass).  Expert-major, token-ascending order is this library's
 * reading, chosen so the result is unique. */
MX_API int moe_permute(const int32_t* topk_ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                int32_t* sorted_slot, void* ws, size_t ws_bytes, mx_stream_t stream);

/* moe_permute without a caller workspace.  The pages have no counterpart:
 * this entry exists for callers that are not allowed to allocate device
 * memory (for example a plugin whose host framework owns all device memory
 * and forbids cudaMalloc in its enqueue path, or a serving loop that must not
 * call cudaMalloc because it can synchronise the device).  It computes exactly
 * what moe_permute computes, using a fixed 400 KiB scratch array inside the
 * library that every GPU loading the library keeps until the process exits.
 *  - Limit: the scratch moe_permute_workspace_size(T, E, k) reports must fit
 *    in 400 KiB (T <= 8192, E <= 512, k <= 8 always fits); larger requests
 *    return MX_ERR_WORKSPACE and enqueue nothing.
 *  - The array is shared by every call on a device and keeps the last call's
 *    contents; calls that overlap on the GPU race, so keep them on one stream.
 *  - The first call on a device looks up the array's device address; make it
 *    before any stream capture.  The address is kept per device and CUDA
 *    context: after cudaDeviceReset the next call looks it up again.
 *    Device-side id errors are not reported.
 *  - Allocates nothing: no cudaMalloc/cudaFree or allocating library call. */
MX_API int moe_permute_no_alloc(const int32_t* topk_ids, int T, int E, int k, int32_t* counts,
                                int32_t* offsets, int32_t* sorted_slot, mx_stream_t stream);

/* Bytes of a prepared (kernel-layout) weight table.  which = 1: W1, the
 * gate/up projection [E1][2I][H] (rows 0..I-1 gate, I..2I-1 up); which = 2:
 * W2, the down projection [E1][H][I].  E1 = E + 1 experts (shared last). */
MX_API size_t moe_prepared_weight_bytes(int E1, int H, int I, int fmt, int which);

/* Load-time re-layout of a canonical MX weight table into the kernel layout
 * (done once per weight set, off the serving path).
 *   codes  [E1][rows][K] (E4M3) or [E1][rows][K/2] (E2M1), scales [E1][rows][K/32],
 *   rows/K = 2I/H for which = 1 and H/I for which = 2.
 *   dst: moe_prepared_weight_bytes(...) bytes, 256-byte aligned.
 * Errors: MX_ERR_INVALID_ARG, MX_ERR_UNSUPPORTED (H or I not a multiple of
 * 128), MX_ERR_ALIGNMENT, MX_ERR_WORKSPACE (dst_bytes too small).
 * Source: the MI355X page, the passage after Figure 4 (MXFP8 weight and scale
 * re-layout moved to model load; serving uses the prepared form directly). */
MX_API int moe_prepare_weights(const uint8_t* codes, const uint8_t* scales, int E1, int H, int I, int fmt,
                        int which, void* dst, size_t dst_bytes, mx_stream_t stream);

/* Bytes of workspace the two grouped GEMM calls need. */
MX_API size_t moe_gemm_workspace_size(int T, int H, int I, int E, int k);

/* Grouped gate/up GEMM with SwiGLU and MXFP8 re-quantisation of h fused into
 * the epilogue.  For every slot position p (expert e = the segment of
 * `offsets` holding p, token t = sorted_slot[p] / (k+1)):
 *   g_i = sum_h act[t,h] Wg[e,i,h],  u_i = sum_h act[t,h] Wu[e,i,h]  (fp32 accumulation
 *   of exactly decoded MX products), h_i = silu(g_i) * u_i, then h quantised
 *   per 32 along I exactly as mx_quantize_act does.
 *   act_codes/act_scales: MXFP8 activations [T, H], [T, H/32].
 *   offsets/sorted_slot: moe_permute output.  w1_prep: moe_prepare_weights(which=1).
 *   h_codes [T*(k+1), I], h_scales [T*(k+1), I/32]: row p = slot position p.
 * fp32 accumulation means an h code next to a rounding boundary may differ by
 * one step from an exact-arithmetic reference.
 * Errors: MX_ERR_INVALID_ARG, MX_ERR_UNSUPPORTED (H or I % 128, E > 1024),
 * MX_ERR_ALIGNMENT, MX_ERR_WORKSPACE, MX_ERR_CUDA.
 * Source: the MI355X page, Figure 3 and its passage (separate small-M and
 * large-M launchers, tiles chosen from the local shape, grouped programs
 * reordered for cache reuse), Figure 4 (routed and shared experts in one
 * grouped GEMM) and the correctness passage (packed gate/up slices, SwiGLU). */
MX_API int moe_grouped_gemm_swiglu(const uint8_t* act_codes, const uint8_t* act_scales,
                            const int32_t* offsets, const int32_t* sorted_slot, const void* w1_prep,
                            int fmt, int T, int H, int I, int E, int k, uint8_t* h_codes,
                            uint8_t* h_scales, void* ws, size_t ws_bytes, mx_stream_t stream);

/* Grouped down GEMM with the weighted scatter-combine fused into the epilogue:
 *   out[t, :] += w_s * sum_i h[p,i] Wd[e,:,i]   (w_s = topk_w[t,j] for a routed
 *   slot, 1 for the shared slot), fp32 atomic adds into `out`.
 *   out [T, H] fp32 must be zero-filled (or hold a residual) by the caller.
 * Errors: as moe_grouped_gemm_swiglu.
 * Source: the Kimi K3 page, section on moving the MXFP4 top-k finalize into
 * the epilogue (one launch and one intermediate write/read removed); the
 * MI355X page, Figure 4 (the shared expert's output added with the routed
 * ones). */
MX_API int moe_grouped_gemm_down_combine(const uint8_t* h_codes, const uint8_t* h_scales,
                                  const int32_t* offsets, const int32_t* sorted_slot,
                                  const float* topk_w, const void* w2_prep, int fmt, int T, int H,
                                  int I, int E, int k, float* out, void* ws, size_t ws_bytes,
                                  mx_stream_t stream);


/* Bytes of workspace moe_forward needs (intermediates + GEMM scratch). */
MX_API size_t moe_workspace_size(int T, int H, int I, int E, int k, int fmt);

/* The whole layer in one call, no host synchronisation: quantise, route,
 * permute, both grouped GEMMs; out [T, H] fp32 is overwritten.  Three kernel
 * launches: a prologue (routing, quantisation, zeroing of out, the
 * permutation and, on the wide schedule, the activation rows in slot order;
 * for more than 256 tokens its phases are separated by grid barriers, plus
 * two 4-byte memsets of its counters) and the two grouped GEMMs (up to 256
 * tokens as programmatically dependent launches).  A batch whose prologue grid
 * would not fit on the GPU at once falls back to separate permutation launches.
 * Errors: union of the step calls.
 * Source: the MI355X page, the passage on launch cost and graph execution and
 * Figure 4's passage (removing launches and intermediate traffic raised output
 * throughput most at concurrency 1); the Ling-3.0-flash page, on kernel nodes
 * of 1.5-6 us each whose launch floor is comparable to their arithmetic. */
MX_API int moe_forward(const void* x_bf16, const float* logits, const void* w1_prep, const void* w2_prep,
                int fmt, int T, int H, int I, int E, int k, float* out, void* ws, size_t ws_bytes,
                mx_stream_t stream);

/* Number of kernel launches moe_forward enqueues for this shape on the
 * current device (host only: no kernel runs; -1 for a shape moe_forward
 * rejects, 0 for T = 0). */
MX_API int moe_forward_launches(int T, int H, int I, int E, int k, int fmt);

/* ---- layer variants ---- */
#define MX_ACT_SWIGLU 0      /* h = silu(g) * u */
#define MX_ACT_SWIGLU_OAI 1  /* h = g' * sigmoid(alpha * g') * (u' + 1), g' = min(g, limit), u' = clamp(u, +-limit) */
#define MX_SHARED_FOLDED 0   /* shared expert as a routed-table slot every token selects */
#define MX_SHARED_DENSE 1    /* shared expert as its own dense MLP launches */

/* Options of the layer variants (a NULL pointer means the defaults: SwiGLU,
 * folded shared expert, MXFP8 activations).
 *  - activation: MX_ACT_SWIGLU or MX_ACT_SWIGLU_OAI.  SwiGLU-OAI follows the
 *    MI355X page's correctness passage (the model's SwiGLU-OAI parameters are
 *    passed into the MoE); the page gives no values, the caller does: alpha
 *    (the sigmoid slope) and limit (> 0; the gate is clamped above at limit,
 *    the up projection to [-limit, limit]).
 *  - shared_expert: MX_SHARED_FOLDED (the MI355X page's Figure 4: one grouped
 *    GEMM pair covers routed and shared experts) or MX_SHARED_DENSE (the path
 *    that figure replaces: the shared expert runs as its own dense gate/up and
 *    down launches after the routed ones; same arithmetic, two more launches).
 *  - act_fmt: MX_E4M3 (MXFP8 activations and h) or MX_E2M1 (MXFP4
 *    activations and h: x and h are quantised to E2M1 with an E8M0 scale per
 *    32 elements, emax 2, and both grouped GEMMs run on the packed-FP4 MMA
 *    with MXFP4 weights on both sides).  MX_E2M1 needs fmt == MX_E2M1
 *    (MX_ERR_UNSUPPORTED with MXFP8 weights).  The activation codes
 *    (and h codes) are then [rows, K/2] bytes, element 2i in the low nibble.
 *    Source: the MI355X page's opening results list (an MXFP4 model) and its
 *    passage on native MX back ends; the element and scale rule is OCP MX
 *    v1.0's for E2M1. */
typedef struct mx_layer_opts {
  int activation;
  float alpha;
  float limit;
  int shared_expert;
  int act_fmt;
} mx_layer_opts;

/* moe_forward with layer options (see mx_layer_opts); the workspace size is
 * moe_workspace_size's.  Errors: as moe_forward, plus MX_ERR_INVALID_ARG for
 * an unknown option value or a non-positive / non-finite limit. */
MX_API int moe_forward_ex(const void* x_bf16, const float* logits, const void* w1_prep, const void* w2_prep,
                          int fmt, int T, int H, int I, int E, int k, float* out, void* ws, size_t ws_bytes,
                          const mx_layer_opts* opts, mx_stream_t stream);

/* moe_grouped_gemm_swiglu with layer options (the activation and act_fmt are
 * used: with MX_E2M1 the activation codes are MXFP4 [T, H/2] bytes and h is
 * written as MXFP4, [rows, I/2] bytes; shared_expert must be folded). */
MX_API int moe_grouped_gemm_swiglu_ex(const uint8_t* act_codes, const uint8_t* act_scales,
                                      const int32_t* offsets, const int32_t* sorted_slot, const void* w1_prep,
                                      int fmt, int T, int H, int I, int E, int k, uint8_t* h_codes,
                                      uint8_t* h_scales, void* ws, size_t ws_bytes, const mx_layer_opts* opts,
                                      mx_stream_t stream);

/* moe_grouped_gemm_down_combine with layer options: act_fmt MX_E2M1 reads
 * MXFP4 h ([rows, I/2] bytes; needs MXFP4 weights); the other fields must hold
 * their defaults' kind (the activation is not used here). */
MX_API int moe_grouped_gemm_down_combine_ex(const uint8_t* h_codes, const uint8_t* h_scales,
                                            const int32_t* offsets, const int32_t* sorted_slot,
                                            const float* topk_w, const void* w2_prep, int fmt, int T, int H,
                                            int I, int E, int k, float* out, void* ws, size_t ws_bytes,
                                            const mx_layer_opts* opts, mx_stream_t stream);

/* Kernel launches moe_forward_ex enqueues for this shape and these options
 * (host only; -1 for a rejected shape or option). */
MX_API int moe_forward_launches_ex(int T, int H, int I, int E, int k, int fmt, const mx_layer_opts* opts);

/* Copy the workspace status word to *host_status (synchronising `stream`) and
 * clear it.  0 = no device-side error; otherwise an MX_ERR_* code. */
MX_API int moe_get_status(void* ws, mx_stream_t stream, int* host_status);

/* Test hook: the wall-clock limit, in nanoseconds, of every bounded wait inside
 * the GEMM kernels (default 2e9).  A tiny limit makes the waits run out, which
 * exercises the MX_ERR_TIMEOUT path without hanging the GPU. */
MX_API void mx_debug_set_wait_limit_ns(uint64_t ns);

/* Measurement hook: while enabled (enable != 0), each grouped-GEMM kernel
 * launch is bracketed by two CUDA events the library records on the launch's
 * stream (the first 4096 launches after enabling; events of the device that is
 * current at the first recorded launch, later launches on another device are
 * not recorded).  mx_debug_gemm_times waits for the recorded events, writes for
 * the first min(n, max) launches the kernel's device time in milliseconds
 * (ms[i]) and its epilogue (epi[i]: 0 gate/up, 1 down), forgets them and
 * returns n, the number recorded (-1: a CUDA error).  Enabling or disabling
 * also forgets them.  Not for streams being captured into a CUDA graph.  The
 * pages have no counterpart: it times the dominant kernel apart from the row
 * gather that shares its call. */
MX_API void mx_debug_time_gemms(int enable);
MX_API int mx_debug_gemm_times(float* ms, int* epi, int max);

/* Hash of the sources, flags and compiler this library was built from
 * (16 hex digits; static string).  Lets a caller check that the library it
 * loaded was compiled from the sources it expects. */
MX_API const char* mx_build_stamp(void);

#ifdef __cplusplus
}
#endif
#endif /* MXMOE_H_ */
