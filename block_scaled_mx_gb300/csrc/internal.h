// Internal launcher interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Launchers only enqueue work; argument checks happen in
// api.cu.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mxk {

// ---- prep.cu
// x bf16 -> MX codes (fmt MX_E4M3: one byte per element; MX_E2M1: two per byte)
cudaError_t launch_quantize_act(const void* x, int64_t n_elems, uint8_t* codes, uint8_t* scales,
                                cudaStream_t s, int fmt = 0 /* MX_E4M3 */);
cudaError_t launch_quantize_weights(const float* w, int64_t n_elems, int fmt, uint8_t* codes,
                                    uint8_t* scales, cudaStream_t s);
cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                        cudaStream_t s);

// Scratch of the permutation: status word, chunk histograms, per-slot local
// ranks, chunk bases and the last-block counter.
struct PermuteScratch {
  int* status;
  int* chunk_counts;   // [nchunks][E]
  int* chunk_base;     // [nchunks][E]
  int* local_rank;     // [T*k]
  unsigned* done;      // 1 counter
};
constexpr int kPermuteChunk = 256;
size_t permute_scratch_bytes(int T, int E, int k);
PermuteScratch permute_scratch_carve(void* ws, int T, int E, int k);
cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* sorted_slot, const PermuteScratch& sc,
                           cudaStream_t s);

// The fused layer's first launch: routing, activation quantisation and zeroing
// of out over all blocks; with `permute` (T <= kPermuteChunk) the last block
// also computes counts / offsets / sorted_slot.
struct PrologueArgs {
  const uint4* x;       // bf16 [T, H] as 16-byte groups
  int64_t n8;           // T*H/8
  uint2* codes;         // MXFP8 codes, 8 per group (MXFP4: 4 bytes per group)
  int act_e2m1;         // quantise to MXFP4 instead
  uint8_t* scales;
  const float* logits;
  int T, E, k;
  int32_t* ids;
  float* topk_w;
  float4* out;
  int64_t n_out4;       // T*H/4
  int permute;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_slot;
  PermuteScratch sc;
};
cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t s);
// The prologue of a batch larger than one permutation chunk in one launch:
// routing, quantisation, zeroing, the chunked permutation and (gathered set)
// the activation rows in slot order, phases separated by grid barriers.
struct BigPrologueArgs {
  unsigned* bar;            // grid-barrier counter (zeroed by the launch)
  uint8_t* gathered;        // [T*(k+1), row_bytes] slot-ordered activation rows, or null
  int64_t row_bytes;        // bytes of one activation row (H, or H/2 for MXFP4)
  uint32_t* gathered_scales;  // [H/128][T*(k+1)] their scales, K-chunk-major (with gathered)
  int64_t scale_words;      // H/128: 32-bit scale words of one activation row
  unsigned long long wait_limit_ns;
};
int prologue_big_blocks(const PrologueArgs& a);  // 0: not possible on this GPU
cudaError_t launch_prologue_big(const PrologueArgs& a, const BigPrologueArgs& b, int blocks, cudaStream_t s);

// dst[p, :] = src[sorted_slot[p] / (k+1), :] for p < n_rows (rows of `row_bytes`),
// and the rows' scales K-chunk-major: dst_sc[c * n_rows + p] = word c of scale
// row sorted_slot[p] / (k+1) of src_sc ([T, scale_words] 32-bit words, one per
// 128-element K chunk).
cudaError_t launch_gather_rows(const uint8_t* src, int T, int64_t row_bytes,
                               const int32_t* sorted_slot, int k, int n_rows, uint8_t* dst,
                               const uint32_t* src_sc, int64_t scale_words, uint32_t* dst_sc,
                               int* status, cudaStream_t s);

// Kernel layout of one weight table (see gemm.cu): codes in 128-row x
// 128-element blocks, block (e, rb, kc) at ((e*RB + rb)*NK + kc); scales in
// 512-byte blocks in the tensor-memory order of the block-scaled MMA.
struct PreparedLayout {
  int E1, rows, K, fmt;
  int RB, NK;
  int interleave;           // W1: prepared row block 2m is gate block m, 2m + 1 is up block m
  size_t block_code_bytes;  // 16384 (E4M3) or 8192 (E2M1)
  size_t codes_bytes, scales_offset, scales_bytes, total_bytes;
};
PreparedLayout prepared_layout(int E1, int rows, int K, int fmt, int interleave);
cudaError_t launch_prepare_weights(const uint8_t* codes, const uint8_t* scales,
                                   const PreparedLayout& L, uint8_t* dst, cudaStream_t s);

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s);

// ---- router.cu
struct RouterArgs {
  const void* x;         // bf16 [T, H]
  const void* w;         // bf16 [E, H]
  const float* bias;     // [E] or null
  int T, H, E, k;
  float* logits;         // [T, E] or null
  int32_t* ids;          // [T, k] or null (logits only)
  float* topk_w;         // [T, k]
  int* status;
  uint64_t wait_limit_ns;
  unsigned* counter;        // a word of the workspace: blocks finished (small batches; zero between calls)
  float* scratch_logits;    // [T, E] in the workspace when the caller keeps no logits, or null
};
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);

// ---- gemm.cu
struct GemmArgs {
  int epi;               // 0: gate/up + SwiGLU + requant, 1: down + combine
  int fmt;               // weight format (MX_E4M3 / MX_E2M1)
  int T, H, I, E, k;
  const void* w_prep;    // prepared weights
  const uint8_t* b_codes;   // gather4: activation codes [T, H] (rows gathered by token);
                            // else rows [n_rows, K] already in slot order
  int gather4;
  int n_rows;               // T*(k+1)
  const uint8_t* b_scales;  // GEMM1: act scales [T, H/32] by token; GEMM2: h scales [rows, I/32]
  const uint32_t* b_scales_t;  // GEMM1 on gathered rows: their scales K-chunk-major
                               // [H/128][n_rows] (one word per row and chunk), or null
  const int32_t* offsets;   // [E+2]
  const int32_t* sorted_slot;
  const float* topk_w;      // GEMM2
  uint8_t* h_codes;         // GEMM1 out
  uint8_t* h_scales;        // GEMM1 out
  float* out;               // GEMM2 out
  int* status;
  int bn;                   // token-tile width (16 .. 224; a pair's tile spans both CTAs)
  uint64_t wait_limit_ns;
  // programmatic dependent launch: 0 none; 1 the previous grid produced the
  // offsets and the B rows (wait before anything); 2 the previous grid produced
  // only the B rows and their scales (weights stream before the wait)
  int pdl;
  // run as clusters of two CTAs with the pair MMA (M = 256 over two SMs; each
  // SM loads half of the token rows); needs pair_supported()
  int pair;
  // down GEMM: one W2 row block per tile (M = 128) instead of two, so that a
  // wide token tile still has two accumulator buffers
  int one_blk;
  // expert window: this launch covers n_exp experts (0: all E + 1), table
  // experts e_base .. e_base + n_exp - 1; `offsets` then points at entry e_base
  int n_exp, e_base;
  // gate/up epilogue activation: 0 SwiGLU, 1 SwiGLU-OAI with alpha and limit
  int act;
  float alpha, limit;
  // MXFP4 weights with MXFP4 token rows (kind::mxf4): activations / h packed
  // E2M1 ([rows, K/2] bytes), h re-quantised to MXFP4 by the gate/up epilogue
  int a4;
};
bool pair_supported(const GemmArgs& a);
// Per-launch timing of the grouped GEMM kernels (mx_debug_time_gemms).
void gemm_timing_enable(bool on);
int gemm_timing_read(float* ms, int* epi, int max);

cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t s);

}  // namespace mxk
