// C ABI of libmxmoe.so: argument validation, workspace carving and the
// orchestration of the MX MoE expert layer (see include/mxmoe.h).
#include <cuda_runtime.h>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/mxmoe.h"
#include "internal.h"

using namespace mxk;

namespace {

uint64_t g_wait_limit_ns = 2000000000ull;

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t al256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MX_OK : MX_ERR_CUDA; }

// Token-row tile width of the grouped GEMMs, chosen from the mean rows per
// expert (known on the host, no device read).  The narrow decode schedule
// (16 or 32 rows) streams weights with two accumulator buffers; 16-row tiles
// (a few rows per expert) free shared memory for a third pipeline stage at the
// price of a second tile for experts with more rows (the shared expert).  The
// wide prefill schedule reuses each weight tile over many token rows, and an
// SM's operand intake is its limit there, so the tile is as wide as tensor
// memory allows with three pipeline stages of scale factors: 208 rows.  The
// gate/up GEMM then holds one accumulator buffer (2 x 208 columns of g and u),
// the down GEMM two (one W2 row block a tile, M = 128: the atomic-combine
// epilogue overlaps the next tile's MMAs).  On the 8192-token layer 208 beat
// 192 by 4% in each GEMM; 224 leaves room for only two stages and lost.
// `which`: 0 gate/up, 1 down.
int choose_bn(int T, int E, int k, int which) {
  const char* env = std::getenv(which == 1 && std::getenv("MXMOE_BN2") ? "MXMOE_BN2" : "MXMOE_BN");
  if (env) {
    const int v = std::atoi(env);
    if (v >= 16 && v <= 224 && v % 16 == 0) return v;
  }
  const double mean_rows = static_cast<double>(T) * (k + 1) / (E + 1);
  // gate/up: smaller B tiles leave room for a third stage; down: 32 rows (the
  // shared expert's T rows in half the tiles, each reading the expert's W2
  // once more: decode_mxfp4 layer 272 -> 267 us)
  if (mean_rows < 12.0) return which == 1 ? 32 : 16;
  if (mean_rows < 48.0) return 32;
  return 208;
}

int check_gemm_shape(int T, int H, int I, int E, int k, int fmt) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k < 1 || k > E || k > 32) return MX_ERR_INVALID_ARG;
  if (fmt != MX_E4M3 && fmt != MX_E2M1) return MX_ERR_INVALID_ARG;
  if (H % 128 || I % 128 || E > 1024) return MX_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * (k + 1) > INT32_MAX / 2) return MX_ERR_UNSUPPORTED;
  return MX_OK;
}

// The wide schedule can run the grouped GEMMs as CTA pairs (M = 256 MMAs over
// two SMs, each loading half of a tile's token rows) when every pair tile has
// its full four weight row blocks.  Measured on the 8192-token prefill layer,
// pairs were slower than single CTAs (gate/up 1.24 vs 1.10 ms: the per-SM
// operand rate did not rise and the pair waits for both epilogues between
// tiles), so they run only when MXMOE_PAIR=1 asks for them (A/B runs, tests).
void choose_pair(GemmArgs& a) {
  const char* env = std::getenv("MXMOE_PAIR");
  a.pair = (!a.gather4 && env && env[0] == '1' && pair_supported(a)) ? 1 : 0;
}

// The narrow schedule gathers each tile's few token rows with TMA gather4; the
// wide schedule first copies the activation rows into slot order (one row-gather
// kernel) so that each stage's 128 token rows arrive as one TMA box.
bool wide_schedule(int T, int E, int k) { return choose_bn(T, E, k, 0) > 64; }

// The wide schedule's slot-ordered activation rows (H bytes each) followed by
// their scales K-chunk-major (H/128 words per row).
size_t gather_bytes(int T, int H, int E, int k) {
  const size_t slots = static_cast<size_t>(T) * (k + 1);
  return wide_schedule(T, E, k) ? al256(slots * H) + al256(slots * (H / 32)) : 0;
}
uint32_t* gathered_scales(uint8_t* act_sorted, int T, int H, int k) {
  return reinterpret_cast<uint32_t*>(act_sorted + al256(static_cast<size_t>(T) * (k + 1) * H));
}

// Kernel launches moe_forward enqueues for a shape (mirrors its branches):
// the prologue; the chunked permutation when the prologue cannot permute
// (count + scatter, or count alone for one chunk); the row gather of the wide
// schedule; the two grouped GEMMs.
int forward_launches(int T, int E, int k, bool dense_shared = false) {
  const bool wide = wide_schedule(T, E, k);
  const bool fused = T <= kPermuteChunk && !wide;
  const int nchunks = (T + kPermuteChunk - 1) / kPermuteChunk;
  const char* sep = std::getenv("MXMOE_SEPARATE_PERMUTE");
  if (!fused && !(sep && sep[0] == '1')) {
    // the one-launch prologue of a large batch, when its grid fits on this GPU
    PrologueArgs pa{};
    pa.T = T;
    pa.E = E;
    pa.k = k;
    if (prologue_big_blocks(pa) > 0) return 1 + (dense_shared ? 4 : 2);
  }
  return 1 + (fused ? 0 : (nchunks > 1 ? 2 : 1)) + (wide ? 1 : 0) + (dense_shared ? 4 : 2);
}

// moe_forward workspace carve (status word first, shared with the permutation
// scratch).
struct ForwardWs {
  PermuteScratch perm;
  int32_t* ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_slot;
  uint8_t* act_codes;
  uint8_t* act_scales;
  uint8_t* act_sorted;
  uint8_t* h_codes;
  uint8_t* h_scales;
  unsigned* gbar;  // grid-barrier counter of the large-batch prologue
  size_t bytes;
};

ForwardWs carve_forward(void* ws, int T, int H, int I, int E, int k) {
  ForwardWs f{};
  uint8_t* p = static_cast<uint8_t*>(ws);
  size_t off = 0;
  const size_t slots = static_cast<size_t>(T) * (k + 1);
  auto take = [&](size_t b) {
    uint8_t* r = p ? p + off : nullptr;
    off += al256(b);
    return r;
  };
  uint8_t* perm = take(permute_scratch_bytes(T, E, k));
  if (p) f.perm = permute_scratch_carve(perm, T, E, k);
  f.ids = reinterpret_cast<int32_t*>(take(static_cast<size_t>(T) * k * 4));
  f.topk_w = reinterpret_cast<float*>(take(static_cast<size_t>(T) * k * 4));
  f.counts = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E + 1) * 4));
  f.offsets = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E + 2) * 4));
  f.sorted_slot = reinterpret_cast<int32_t*>(take(slots * 4));
  f.act_codes = take(static_cast<size_t>(T) * H);
  f.act_scales = take(static_cast<size_t>(T) * (H / 32));
  f.act_sorted = take(gather_bytes(T, H, E, k));
  f.h_codes = take(slots * I);
  f.h_scales = take(slots * (I / 32));
  f.gbar = reinterpret_cast<unsigned*>(take(4));
  f.bytes = off;
  return f;
}

// The layer options, checked and with defaults filled in.
struct LayerOpts {
  int act = MX_ACT_SWIGLU;
  float alpha = 1.0f, limit = 0.0f;
  int shared = MX_SHARED_FOLDED;
  int act_fmt = MX_E4M3;
};

int read_opts(const mx_layer_opts* o, LayerOpts* out) {
  LayerOpts r;
  if (o) {
    if (o->activation != MX_ACT_SWIGLU && o->activation != MX_ACT_SWIGLU_OAI) return MX_ERR_INVALID_ARG;
    if (o->shared_expert != MX_SHARED_FOLDED && o->shared_expert != MX_SHARED_DENSE) return MX_ERR_INVALID_ARG;
    if (o->act_fmt != MX_E4M3 && o->act_fmt != MX_E2M1) return MX_ERR_INVALID_ARG;
    if (o->activation == MX_ACT_SWIGLU_OAI && !(o->limit > 0.0f && o->limit <= 3.0e38f && o->alpha == o->alpha &&
                                                 o->alpha > -3.0e38f && o->alpha < 3.0e38f))
      return MX_ERR_INVALID_ARG;
    r.act = o->activation;
    r.alpha = o->alpha;
    r.limit = o->limit;
    r.shared = o->shared_expert;
    r.act_fmt = o->act_fmt;
  }
  *out = r;
  return MX_OK;
}

// MXFP4 activations run on kind::mxf4, which needs both operands E2M1: they
// come with MXFP4 weights only.
int check_act_fmt(const LayerOpts& lo, int fmt) {
  return (lo.act_fmt == MX_E2M1 && fmt != MX_E2M1) ? MX_ERR_UNSUPPORTED : MX_OK;
}

// The experts one grouped-GEMM launch covers: n table experts from e_base
// (n = 0: all E + 1).
struct Window {
  int n = 0, e_base = 0;
};

int run_gemm1(const uint8_t* act_codes, const uint8_t* act_scales, const int32_t* offsets,
              const int32_t* sorted_slot, const void* w1_prep, int fmt, int T, int H, int I, int E,
              int k, uint8_t* h_codes, uint8_t* h_scales, int* status, uint8_t* act_sorted,
              cudaStream_t s, int pdl = 0, const LayerOpts& lo = LayerOpts(), Window win = Window(),
              bool gather_rows = true) {
  const int n_rows = T * (k + 1);
  if (n_rows == 0) return MX_OK;
  GemmArgs a{};
  a.bn = choose_bn(T, E, k, 0);
  a.gather4 = a.bn <= 64 ? 1 : 0;
  a.pdl = pdl;
  a.a4 = lo.act_fmt == MX_E2M1 ? 1 : 0;
  a.act = lo.act;
  a.alpha = lo.alpha;
  a.limit = lo.limit;
  a.n_exp = win.n;
  a.e_base = win.e_base;
  if (!a.gather4 && gather_rows) {
    if (launch_gather_rows(act_codes, T, a.a4 ? H / 2 : H, sorted_slot, k, n_rows, act_sorted,
                           reinterpret_cast<const uint32_t*>(act_scales), H / 128,
                           gathered_scales(act_sorted, T, H, k), status, s) != cudaSuccess)
      return MX_ERR_CUDA;
  }
  a.epi = 0;
  a.fmt = fmt;
  a.T = T;
  a.H = H;
  a.I = I;
  a.E = E;
  a.k = k;
  a.w_prep = w1_prep;
  a.b_codes = a.gather4 ? act_codes : act_sorted;
  a.n_rows = n_rows;
  a.b_scales = act_scales;
  a.b_scales_t = a.gather4 ? nullptr : gathered_scales(act_sorted, T, H, k);
  a.offsets = offsets + win.e_base;
  a.sorted_slot = sorted_slot;
  a.h_codes = h_codes;
  a.h_scales = h_scales;
  a.status = status;
  a.wait_limit_ns = g_wait_limit_ns;
  choose_pair(a);
  return cuda_status(launch_grouped_gemm(a, s));
}

int run_gemm2(const uint8_t* h_codes, const uint8_t* h_scales, const int32_t* offsets,
              const int32_t* sorted_slot, const float* topk_w, const void* w2_prep, int fmt, int T,
              int H, int I, int E, int k, float* out, int* status, cudaStream_t s, int pdl = 0,
              Window win = Window(), int a4 = 0) {
  const int n_rows = T * (k + 1);
  if (n_rows == 0) return MX_OK;
  GemmArgs a{};
  a.epi = 1;
  a.fmt = fmt;
  a.T = T;
  a.H = H;
  a.I = I;
  a.E = E;
  a.k = k;
  a.w_prep = w2_prep;
  a.b_codes = h_codes;
  a.n_rows = n_rows;
  a.b_scales = h_scales;
  a.offsets = offsets + win.e_base;
  a.n_exp = win.n;
  a.e_base = win.e_base;
  a.sorted_slot = sorted_slot;
  a.topk_w = topk_w;
  a.out = out;
  a.status = status;
  a.pdl = pdl;
  a.a4 = a4;
  a.bn = choose_bn(T, E, k, 1);
  // wide tiles take one W2 row block each (two accumulator buffers fit); MXFP4
  // activations keep two row blocks of 96 rows
  if (a4 && a.bn > 96) a.bn = 96;
  a.one_blk = (!a4 && a.bn >= 128) ? 1 : 0;
  a.wait_limit_ns = g_wait_limit_ns;
  choose_pair(a);
  return cuda_status(launch_grouped_gemm(a, s));
}

}  // namespace

extern "C" {

const char* mx_status_string(int status) {
  switch (status) {
    case MX_OK: return "ok";
    case MX_ERR_INVALID_ARG: return "invalid argument";
    case MX_ERR_UNSUPPORTED: return "unsupported shape or format";
    case MX_ERR_ALIGNMENT: return "pointer not sufficiently aligned";
    case MX_ERR_WORKSPACE: return "workspace or destination too small";
    case MX_ERR_CUDA: return "CUDA error";
    case MX_ERR_TIMEOUT: return "device wait timed out";
    case MX_ERR_DEVICE_ARG: return "device-side index out of range";
    default: return "unknown status";
  }
}

int mx_quantize_act(const void* x_bf16, int T, int H, uint8_t* codes, uint8_t* scales,
                    mx_stream_t stream) {
  if (T < 0 || H <= 0) return MX_ERR_INVALID_ARG;
  if (T == 0) return MX_OK;
  if (!x_bf16 || !codes || !scales) return MX_ERR_INVALID_ARG;
  if (H % 32) return MX_ERR_UNSUPPORTED;
  if (!aligned(x_bf16, 16) || !aligned(codes, 16)) return MX_ERR_ALIGNMENT;
  return cuda_status(launch_quantize_act(x_bf16, static_cast<int64_t>(T) * H, codes, scales,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int mx_quantize_act_ex(const void* x_bf16, int T, int H, int fmt, uint8_t* codes, uint8_t* scales,
                       mx_stream_t stream) {
  if (T < 0 || H <= 0 || (fmt != MX_E4M3 && fmt != MX_E2M1)) return MX_ERR_INVALID_ARG;
  if (T == 0) return MX_OK;
  if (!x_bf16 || !codes || !scales) return MX_ERR_INVALID_ARG;
  if (H % 32) return MX_ERR_UNSUPPORTED;
  if (!aligned(x_bf16, 16) || !aligned(codes, 16)) return MX_ERR_ALIGNMENT;
  return cuda_status(launch_quantize_act(x_bf16, static_cast<int64_t>(T) * H, codes, scales,
                                         reinterpret_cast<cudaStream_t>(stream), fmt));
}

int mx_quantize_weights(const float* w, int64_t rows, int K, int fmt, uint8_t* codes,
                        uint8_t* scales, mx_stream_t stream) {
  if (rows < 0 || K <= 0 || (fmt != MX_E4M3 && fmt != MX_E2M1)) return MX_ERR_INVALID_ARG;
  if (rows == 0) return MX_OK;
  if (!w || !codes || !scales) return MX_ERR_INVALID_ARG;
  if (K % 32) return MX_ERR_UNSUPPORTED;
  if (!aligned(w, 16) || !aligned(codes, 16)) return MX_ERR_ALIGNMENT;
  return cuda_status(launch_quantize_weights(w, rows * K, fmt, codes, scales,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int moe_route_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                   mx_stream_t stream) {
  if (T < 0 || E <= 0 || k < 1 || k > E || k > 32) return MX_ERR_INVALID_ARG;
  if (E > 1024) return MX_ERR_UNSUPPORTED;
  if (T == 0) return MX_OK;
  if (!logits || !topk_ids || !topk_w) return MX_ERR_INVALID_ARG;
  return cuda_status(launch_topk(logits, T, E, k, topk_ids, topk_w, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_permute_workspace_size(int T, int E, int k) {
  if (T < 0 || E <= 0 || k < 1) return 0;
  return permute_scratch_bytes(T, E, k);
}

int moe_permute(const int32_t* topk_ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                int32_t* sorted_slot, void* ws, size_t ws_bytes, mx_stream_t stream) {
  if (T < 0 || E <= 0 || k < 1 || k > E || k > 32) return MX_ERR_INVALID_ARG;
  if (E > 1024) return MX_ERR_UNSUPPORTED;
  if (!counts || !offsets || !ws || (T > 0 && (!topk_ids || !sorted_slot))) return MX_ERR_INVALID_ARG;
  if (ws_bytes < permute_scratch_bytes(T, E, k)) return MX_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return MX_ERR_ALIGNMENT;
  const PermuteScratch sc = permute_scratch_carve(ws, T, E, k);
  return cuda_status(launch_permute(topk_ids, T, E, k, counts, offsets, sorted_slot, sc,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_prepared_weight_bytes(int E1, int H, int I, int fmt, int which) {
  if (E1 <= 0 || H <= 0 || I <= 0 || (fmt != MX_E4M3 && fmt != MX_E2M1)) return 0;
  if (H % 128 || I % 128) return 0;
  if (which == 1) return prepared_layout(E1, 2 * I, H, fmt, 1).total_bytes;
  if (which == 2) return prepared_layout(E1, H, I, fmt, 0).total_bytes;
  return 0;
}

int moe_prepare_weights(const uint8_t* codes, const uint8_t* scales, int E1, int H, int I, int fmt,
                        int which, void* dst, size_t dst_bytes, mx_stream_t stream) {
  if (E1 <= 0 || H <= 0 || I <= 0 || (fmt != MX_E4M3 && fmt != MX_E2M1) || (which != 1 && which != 2))
    return MX_ERR_INVALID_ARG;
  if (!codes || !scales || !dst) return MX_ERR_INVALID_ARG;
  if (H % 128 || I % 128) return MX_ERR_UNSUPPORTED;
  if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(dst, 256)) return MX_ERR_ALIGNMENT;
  const PreparedLayout L =
      which == 1 ? prepared_layout(E1, 2 * I, H, fmt, 1) : prepared_layout(E1, H, I, fmt, 0);
  if (dst_bytes < L.total_bytes) return MX_ERR_WORKSPACE;
  return cuda_status(launch_prepare_weights(codes, scales, L, static_cast<uint8_t*>(dst),
                                            reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_gemm_workspace_size(int T, int H, int I, int E, int k) {
  if (check_gemm_shape(T, H, I, E, k, MX_E4M3) != MX_OK) return 0;
  return al256(256) + gather_bytes(T, H, E, k);
}

int moe_grouped_gemm_swiglu(const uint8_t* act_codes, const uint8_t* act_scales,
                            const int32_t* offsets, const int32_t* sorted_slot, const void* w1_prep,
                            int fmt, int T, int H, int I, int E, int k, uint8_t* h_codes,
                            uint8_t* h_scales, void* ws, size_t ws_bytes, mx_stream_t stream) {
  return moe_grouped_gemm_swiglu_ex(act_codes, act_scales, offsets, sorted_slot, w1_prep, fmt, T, H, I, E, k,
                                    h_codes, h_scales, ws, ws_bytes, nullptr, stream);
}

int moe_grouped_gemm_swiglu_ex(const uint8_t* act_codes, const uint8_t* act_scales,
                               const int32_t* offsets, const int32_t* sorted_slot, const void* w1_prep,
                               int fmt, int T, int H, int I, int E, int k, uint8_t* h_codes,
                               uint8_t* h_scales, void* ws, size_t ws_bytes, const mx_layer_opts* opts,
                               mx_stream_t stream) {
  LayerOpts lo;
  int st = read_opts(opts, &lo);
  if (st != MX_OK) return st;
  if (lo.shared != MX_SHARED_FOLDED) return MX_ERR_INVALID_ARG;
  st = check_gemm_shape(T, H, I, E, k, fmt);
  if (st != MX_OK) return st;
  st = check_act_fmt(lo, fmt);
  if (st != MX_OK) return st;
  if (!offsets || !w1_prep || !ws) return MX_ERR_INVALID_ARG;
  if (T == 0) return MX_OK;
  if (!act_codes || !act_scales || !sorted_slot || !h_codes || !h_scales) return MX_ERR_INVALID_ARG;
  if (!aligned(act_codes, 16) || !aligned(act_scales, 16) || !aligned(h_codes, 16) ||
      !aligned(w1_prep, 256) || !aligned(ws, 256))
    return MX_ERR_ALIGNMENT;
  if (ws_bytes < moe_gemm_workspace_size(T, H, I, E, k)) return MX_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  return run_gemm1(act_codes, act_scales, offsets, sorted_slot, w1_prep, fmt, T, H, I, E, k, h_codes,
                   h_scales, reinterpret_cast<int*>(w), w + al256(256), reinterpret_cast<cudaStream_t>(stream), 0, lo);
}

int moe_grouped_gemm_down_combine(const uint8_t* h_codes, const uint8_t* h_scales,
                                  const int32_t* offsets, const int32_t* sorted_slot,
                                  const float* topk_w, const void* w2_prep, int fmt, int T, int H,
                                  int I, int E, int k, float* out, void* ws, size_t ws_bytes,
                                  mx_stream_t stream) {
  return moe_grouped_gemm_down_combine_ex(h_codes, h_scales, offsets, sorted_slot, topk_w, w2_prep, fmt, T, H, I,
                                          E, k, out, ws, ws_bytes, nullptr, stream);
}

int moe_grouped_gemm_down_combine_ex(const uint8_t* h_codes, const uint8_t* h_scales,
                                     const int32_t* offsets, const int32_t* sorted_slot,
                                     const float* topk_w, const void* w2_prep, int fmt, int T, int H,
                                     int I, int E, int k, float* out, void* ws, size_t ws_bytes,
                                     const mx_layer_opts* opts, mx_stream_t stream) {
  LayerOpts lo;
  int st = read_opts(opts, &lo);
  if (st != MX_OK) return st;
  if (lo.shared != MX_SHARED_FOLDED) return MX_ERR_INVALID_ARG;
  st = check_gemm_shape(T, H, I, E, k, fmt);
  if (st != MX_OK) return st;
  st = check_act_fmt(lo, fmt);
  if (st != MX_OK) return st;
  if (!offsets || !w2_prep || !ws) return MX_ERR_INVALID_ARG;
  if (T == 0) return MX_OK;
  if (!h_codes || !h_scales || !sorted_slot || !topk_w || !out) return MX_ERR_INVALID_ARG;
  if (!aligned(h_codes, 16) || !aligned(h_scales, 16) || !aligned(out, 16) || !aligned(w2_prep, 256) ||
      !aligned(ws, 256))
    return MX_ERR_ALIGNMENT;
  if (ws_bytes < moe_gemm_workspace_size(T, H, I, E, k)) return MX_ERR_WORKSPACE;
  return run_gemm2(h_codes, h_scales, offsets, sorted_slot, topk_w, w2_prep, fmt, T, H, I, E, k, out,
                   reinterpret_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream), 0, Window(),
                   lo.act_fmt == MX_E2M1 ? 1 : 0);
}

size_t moe_workspace_size(int T, int H, int I, int E, int k, int fmt) {
  if (check_gemm_shape(T, H, I, E, k, fmt) != MX_OK) return 0;
  return carve_forward(nullptr, T, H, I, E, k).bytes;
}

int moe_forward(const void* x_bf16, const float* logits, const void* w1_prep, const void* w2_prep,
                int fmt, int T, int H, int I, int E, int k, float* out, void* ws, size_t ws_bytes,
                mx_stream_t stream) {
  return moe_forward_ex(x_bf16, logits, w1_prep, w2_prep, fmt, T, H, I, E, k, out, ws, ws_bytes, nullptr, stream);
}

int moe_forward_ex(const void* x_bf16, const float* logits, const void* w1_prep, const void* w2_prep,
                   int fmt, int T, int H, int I, int E, int k, float* out, void* ws, size_t ws_bytes,
                   const mx_layer_opts* opts, mx_stream_t stream) {
  LayerOpts lo;
  int st = read_opts(opts, &lo);
  if (st != MX_OK) return st;
  st = check_gemm_shape(T, H, I, E, k, fmt);
  if (st != MX_OK) return st;
  st = check_act_fmt(lo, fmt);
  if (st != MX_OK) return st;
  if (T == 0) return MX_OK;
  if (!x_bf16 || !logits || !w1_prep || !w2_prep || !out || !ws) return MX_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(out, 16) || !aligned(w1_prep, 256) || !aligned(w2_prep, 256) ||
      !aligned(ws, 256))
    return MX_ERR_ALIGNMENT;
  if (ws_bytes < moe_workspace_size(T, H, I, E, k, fmt)) return MX_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const ForwardWs f = carve_forward(ws, T, H, I, E, k);
  // Decode sizes run in three launches: the prologue (routing, quantisation,
  // zeroing of out, permutation in its last block), then the two grouped GEMMs
  // as programmatically dependent launches that set up while their predecessor
  // drains.  Larger batches permute in their own chunked kernels.
  const bool fused = T <= kPermuteChunk && !wide_schedule(T, E, k);
  PrologueArgs pa{};
  pa.x = static_cast<const uint4*>(x_bf16);
  pa.n8 = static_cast<int64_t>(T) * H / 8;
  pa.codes = reinterpret_cast<uint2*>(f.act_codes);
  pa.act_e2m1 = lo.act_fmt == MX_E2M1 ? 1 : 0;
  pa.scales = f.act_scales;
  pa.logits = logits;
  pa.T = T;
  pa.E = E;
  pa.k = k;
  pa.ids = f.ids;
  pa.topk_w = f.topk_w;
  pa.out = reinterpret_cast<float4*>(out);
  pa.n_out4 = static_cast<int64_t>(T) * H / 4;
  pa.permute = fused ? 1 : 0;
  pa.counts = f.counts;
  pa.offsets = f.offsets;
  pa.sorted_slot = f.sorted_slot;
  pa.sc = f.perm;
  // A batch larger than one permutation chunk (or on the wide schedule) runs
  // its whole prologue, chunked permutation and row gather included, as one
  // grid-synchronised launch when the grid fits on the GPU at once; else as
  // separate launches.
  const bool wide = wide_schedule(T, E, k);
  // (MXMOE_SEPARATE_PERMUTE=1 forces the separate launches: A/B runs, tests)
  const char* sep = std::getenv("MXMOE_SEPARATE_PERMUTE");
  const int big_blocks = (fused || (sep && sep[0] == '1')) ? 0 : prologue_big_blocks(pa);
  const bool big = big_blocks > 0;
  if (big) {
    BigPrologueArgs b{};
    b.bar = f.gbar;
    b.gathered = wide ? f.act_sorted : nullptr;
    b.row_bytes = lo.act_fmt == MX_E2M1 ? H / 2 : H;
    b.gathered_scales = wide ? gathered_scales(f.act_sorted, T, H, k) : nullptr;
    b.scale_words = H / 128;
    b.wait_limit_ns = g_wait_limit_ns;
    if (launch_prologue_big(pa, b, big_blocks, s) != cudaSuccess) return MX_ERR_CUDA;
  } else {
    if (launch_prologue(pa, s) != cudaSuccess) return MX_ERR_CUDA;
    if (!fused && launch_permute(f.ids, T, E, k, f.counts, f.offsets, f.sorted_slot, f.perm, s) != cudaSuccess)
      return MX_ERR_CUDA;
  }
  // At decode sizes the gate/up GEMM follows the prologue as a programmatic
  // dependent launch and lets the down GEMM launch early (its CTAs take SMs
  // as gate/up CTAs finish and stream their first weight stages).  On the
  // large-batch path the gate/up GEMM starts after the prologue completes and
  // the down GEMM after the gate/up GEMM: there the early down CTAs made the
  // 8192-token layer ~100 us slower (1.93 against 1.82 ms).
  const int pdl1 = fused ? 1 : 0;
  const bool gather = !big;  // the wide schedule's row gather, unless the prologue did it
  if (lo.shared == MX_SHARED_FOLDED) {
    st = run_gemm1(f.act_codes, f.act_scales, f.offsets, f.sorted_slot, w1_prep, fmt, T, H, I, E, k,
                   f.h_codes, f.h_scales, f.perm.status, f.act_sorted, s, pdl1, lo, Window(), gather);
    if (st != MX_OK) return st;
    return run_gemm2(f.h_codes, f.h_scales, f.offsets, f.sorted_slot, f.topk_w, w2_prep, fmt, T, H, I, E,
                     k, out, f.perm.status, s, 2, Window(), lo.act_fmt == MX_E2M1 ? 1 : 0);
  }
  // the shared expert as its own dense MLP: the routed experts' gate/up
  // launch, the shared expert's gate/up launch over all T tokens, then the two
  // down launches (the permutation's shared-slot segment feeds the dense
  // launches, so the arithmetic is the folded layer's)
  Window routed, shared;
  routed.n = E;
  shared.n = 1;
  shared.e_base = E;
  st = run_gemm1(f.act_codes, f.act_scales, f.offsets, f.sorted_slot, w1_prep, fmt, T, H, I, E, k,
                 f.h_codes, f.h_scales, f.perm.status, f.act_sorted, s, pdl1, lo, routed, gather);
  if (st != MX_OK) return st;
  st = run_gemm1(f.act_codes, f.act_scales, f.offsets, f.sorted_slot, w1_prep, fmt, T, H, I, E, k,
                 f.h_codes, f.h_scales, f.perm.status, f.act_sorted, s, pdl1 ? 2 : 0, lo, shared, false);
  if (st != MX_OK) return st;
  st = run_gemm2(f.h_codes, f.h_scales, f.offsets, f.sorted_slot, f.topk_w, w2_prep, fmt, T, H, I, E, k, out,
                 f.perm.status, s, 2, routed, lo.act_fmt == MX_E2M1 ? 1 : 0);
  if (st != MX_OK) return st;
  return run_gemm2(f.h_codes, f.h_scales, f.offsets, f.sorted_slot, f.topk_w, w2_prep, fmt, T, H, I, E, k, out,
                   f.perm.status, s, 2, shared, lo.act_fmt == MX_E2M1 ? 1 : 0);
}

int moe_route_gemm_topk(const void* x_bf16, const void* w_router_bf16, const float* bias, int T, int H, int E,
                        int k, float* logits, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
                        mx_stream_t stream) {
  if (T < 0 || H <= 0 || E <= 0) return MX_ERR_INVALID_ARG;
  const bool select = topk_ids != nullptr || topk_w != nullptr;
  if (select && (!topk_ids || !topk_w || k < 1 || k > E)) return MX_ERR_INVALID_ARG;
  if (!select && !logits) return MX_ERR_INVALID_ARG;
  if (H % 64 || E > 512 || (select && k > 16)) return MX_ERR_UNSUPPORTED;
  if (!ws) return MX_ERR_INVALID_ARG;
  if (ws_bytes < 256) return MX_ERR_WORKSPACE;
  if (T == 0) return MX_OK;
  if (!x_bf16 || !w_router_bf16) return MX_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(w_router_bf16, 16) || !aligned(ws, 256)) return MX_ERR_ALIGNMENT;
  RouterArgs a{};
  a.x = x_bf16;
  a.w = w_router_bf16;
  a.bias = bias;
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = select ? k : 0;
  a.logits = logits;
  a.ids = topk_ids;
  a.topk_w = topk_w;
  a.status = static_cast<int*>(ws);
  a.wait_limit_ns = g_wait_limit_ns;
  // the small-batch kernel's block counter (the workspace's second word) and,
  // when the caller keeps no logits, room for them past the first 256 bytes
  a.counter = static_cast<unsigned*>(ws) + 1;
  if (!logits && ws_bytes >= 256 + static_cast<size_t>(T) * E * sizeof(float))
    a.scratch_logits = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 256);
  return cuda_status(launch_router(a, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_forward_launches(int T, int H, int I, int E, int k, int fmt) {
  return moe_forward_launches_ex(T, H, I, E, k, fmt, nullptr);
}

int moe_forward_launches_ex(int T, int H, int I, int E, int k, int fmt, const mx_layer_opts* opts) {
  LayerOpts lo;
  if (read_opts(opts, &lo) != MX_OK) return -1;
  if (check_gemm_shape(T, H, I, E, k, fmt) != MX_OK) return -1;
  if (T == 0) return 0;
  return forward_launches(T, E, k, lo.shared == MX_SHARED_DENSE);
}

int moe_get_status(void* ws, mx_stream_t stream, int* host_status) {
  if (!ws || !host_status) return MX_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MX_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MX_ERR_CUDA;
  *host_status = v;
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return MX_ERR_CUDA;
  return MX_OK;
}

void mx_debug_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns = ns; }

void mx_debug_time_gemms(int enable) { gemm_timing_enable(enable != 0); }

int mx_debug_gemm_times(float* ms, int* epi, int max) { return gemm_timing_read(ms, epi, max < 0 ? 0 : max); }

#ifndef MXMOE_BUILD_STAMP
#define MXMOE_BUILD_STAMP "unstamped"
#endif
const char* mx_build_stamp(void) { return MXMOE_BUILD_STAMP; }

}  // extern "C"
