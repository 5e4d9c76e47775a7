// Grouped MX block-scaled GEMMs of the MoE expert layer on tcgen05 tensor
// cores (sm_103a), one persistent warp-specialised kernel for both:
//
//   epi 0 (gate/up):  D_gate = Wg[e] . X^T, D_up = Wu[e] . X^T over K = H, then
//                     h = silu(D_gate) * D_up re-quantised to MXFP8 per 32 rows
//                     of I in the epilogue;
//   epi 1 (down):     D = Wd[e] . h^T over K = I, then out[t] += w * D in the
//                     epilogue (fp32 atomic adds: the weighted combine).
//
// Weights are the MMA's A operand (M = 128 rows per sub-tile, two sub-tiles per
// tile), the expert's token rows are the B operand (N = the tile's token count
// rounded up to 16, at most `bn`), so a decode tile with two tokens still runs
// full-width M = 128 MMAs while streaming weights ("swap-AB").  Tiles are
// (expert, token rows, weight rows), expert-major (the down GEMM of a large
// batch runs its weight tiles in groups, one after the other), handed out
// round-robin to one CTA per SM; per-expert token counts are read from the
// device-side permutation offsets, so nothing waits on the host.  A pipeline
// stage is full once its TMA bytes have landed and the scale-staging warps
// have put its scale factors into tensor memory.
//
// Warp roles (448 threads; 576 for the wide gate/up kernel):
//   warp 0      TMA producer: weight blocks (tensor map, 128B swizzle, MXFP4
//               unpacked to the 16-byte-aligned form by the TMA) and token
//               rows (tensor map)
//   warp 1      TMEM allocation; one thread issues
//               tcgen05.mma.kind::mxf8f6f4.block_scale (with a CTA pair:
//               rank 0; rank 1's thread relays its stage completions)
//   warps 2-5   scale staging: the weight and token-row scale factors of
//               every stage, from global memory into every TMEM lane quarter
//               with tcgen05.st
//   warps 6-13  epilogue: tcgen05.ld of the fp32 accumulators, SwiGLU +
//               MXFP8 re-quantisation or weighted combine; warps w, w + 4
//               (and w + 8: warps 6-17 in the wide gate/up kernel) share a TMEM
//               lane quarter (w mod 4) and take its column chunks in turn
// Every wait is bounded (wall clock); a wait that runs out sets
// MX_ERR_TIMEOUT in the status word and every role unwinds.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mxk {

constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;     // with a CTA pair, rank 1's warp relays stage completions
constexpr int kWarpSf0 = 2;     // warps 2..5: TMEM lane quarters 2, 3, 0, 1
constexpr int kWarpEpi0 = 6;    // warps 6..13 (6..17): two (three) per lane quarter
// per epilogue warp, a transpose tile: 16 columns of E4M3 codes (gate/up) or
// 8 columns of fp32 (down)
__host__ __device__ constexpr uint32_t epi_buf_bytes(int epi) { return epi == 0 ? 512u : 1024u; }
constexpr uint32_t kTmemCols = 512;
// per K chunk: SFA of row block 0 (+0), of row block 1 (+8), SFB (+16); a CTA
// pair's CTA has one row block: SFA (+0), SFB (+8)
constexpr uint32_t kSfColsPerChunk = 24;
constexpr uint32_t kSfColsPerChunkPair = 16;
constexpr int kMaxStages = 8;
constexpr int kMaxDevices = 64;

struct GemmParams {
  int epi, afmt, T, H, I, E, k;
  int n_exp, e_base;  // this launch covers n_exp experts, table experts e_base .. e_base + n_exp - 1
  int act;            // gate/up epilogue: 0 SwiGLU, 1 SwiGLU-OAI
  float alpha, limit; // SwiGLU-OAI: sigmoid slope, clamp limit
  int K, NK, NM, RB;
  int MG;  // weight tiles per tile group: groups of MG weight tiles (of every expert and
           // token tile) run one after the other, so the down GEMM's combine targets
           // one slice of `out` at a time (L2-resident atomics).  With a CTA pair,
           // NM and MG count pair tiles (two weight tiles each).
  int bn, stages, acc_bufs;
  int brows;  // token rows one B box loads: bn, or bn / 2 per CTA of a pair
  int n_rows;
  uint32_t a_tx;
  const uint8_t* w_scales;
  const uint8_t* b_scales;
  const uint32_t* b_scales_t;  // gathered rows' scales K-chunk-major [K/128][n_rows], or null
  const int32_t* offsets;
  const int32_t* sorted_slot;
  const float* topk_w;
  uint8_t* h_codes;
  uint8_t* h_scales;
  float* out;
  int* status;
  unsigned long long wait_limit_ns;
  uint32_t off_a, off_b, off_meta, off_bar, off_epi, off_x;
  uint32_t sf_col0;
  uint32_t sfc;     // tensor-memory scale columns per K chunk: 24 (two A blocks), 16 (pair: one)
  uint32_t acc_cols; // accumulator columns per buffer: 2 bn, or bn with a pair
  uint32_t xs;      // pair gate/up: row stride (words) of the exchange buffer
  int gather4;      // B rows gathered by token with TMA gather4 (else one 2-D box of slot rows)
  int pdl;          // see GemmArgs::pdl
  int kps;          // 128-wide K chunks per pipeline stage (1 or 2)
  uint32_t hint_ns; // pair: suspend-time hint of whole-warp barrier waits (0: spin)
  int a4;           // both operands packed E2M1 (kind::mxf4): MXFP4 activations and h
  uint32_t a_slot;  // shared-memory bytes of one K chunk of weight blocks
  uint32_t b_row;   // shared-memory bytes of one token row of one K chunk (128, or 64 packed E2M1)
  int one;          // down GEMM, single CTA: one W2 row block per tile (M = 128), for wide token
                    // tiles with two accumulator buffers
};

struct Tile {
  int e, m, rows, p0;
};

struct Shared {
  uint8_t* base;
  int* offs;     // [E+2]
  int* prefix;   // [E+2] tile prefix
  volatile int* abort_flag;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint64_t* drain;
  uint64_t* exit_bar;  // CTA pair: the peer has finished every role
  uint64_t* peer_full; // CTA pair, rank 0: rank 1's copy of the stage is full
  uint64_t* xfull;     // CTA pair gate/up: the partner has written this CTA's exchange buffer
  uint64_t* xfree;     // CTA pair gate/up: the partner has read its exchange buffer (free to write)
  uint32_t* tmem_slot;
  unsigned* sf_cnt;    // CTA pair: scale warps done with each pipeline slot
  uint32_t rank;       // rank in the CTA pair (0 without one)
  uint32_t hint_ns;    // suspend-time hint of whole-warp waits (0: spin on test_wait)
};

// Tile t -> (group, expert, token tile, weight tile).  Tiles are ordered group-
// major, then expert, token tile and weight tile within the group; prefix[e]
// counts one group's tiles of the experts before e.
__device__ __forceinline__ Tile decode_tile(int t, const Shared& sh, int E, int MG, int bn, int per_group) {
  const int g = t / per_group;
  t -= g * per_group;
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sh.prefix[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  Tile tl;
  tl.e = lo;
  const int local = t - sh.prefix[lo];
  const int nt = local / MG;
  tl.m = g * MG + (local - nt * MG);
  const int cnt = sh.offs[lo + 1] - sh.offs[lo];
  const int n0 = nt * bn;
  tl.rows = min(bn, cnt - n0);
  tl.p0 = sh.offs[lo] + n0;
  return tl;
}

// Abort every role of this CTA (and of the peer CTA of a pair).
template <bool PAIR>
__device__ __forceinline__ void set_abort(const Shared& sh) {
  *sh.abort_flag = 1;
  if (PAIR) st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(sh.abort_flag)), sh.rank ^ 1u), 1u);
}

// Wait that also gives up when another role has aborted.
// SLEEP: poll with a suspend-time hint (whole warps that wait long); the
// single MMA-issuing thread polls without one, to resume the moment a stage
// lands.  PAIR: the barrier also receives arrivals from the peer CTA
// (cluster-scope acquire).
template <bool PAIR, bool SLEEP = true>
__device__ __forceinline__ bool wait_bar(const Shared& sh, uint64_t* bar, uint32_t parity,
                                         unsigned long long limit_ns, int* status) {
  const uint32_t b = smem_u32(bar);
  auto poll = [&](bool sleep) {
    if (PAIR) {
      if (!sleep) return mbar_try_wait_cluster(b, parity);
      return sh.hint_ns ? mbar_try_wait_cluster_sleep(b, parity, sh.hint_ns) : mbar_test_wait_cluster(b, parity);
    }
    return sleep ? mbar_try_wait_sleep(b, parity, 20000u) : mbar_try_wait(b, parity);
  };
  if (poll(false)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (poll(SLEEP)) return true;
    if (*sh.abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      set_status(status, MX_ERR_TIMEOUT);
      set_abort<PAIR>(sh);
      return false;
    }
  }
}

// Whole-warp form of wait_bar: every lane polls, and the outcome is made
// uniform so that the warp leaves (or continues) together.
template <bool PAIR>
__device__ __forceinline__ bool warp_wait_bar(const Shared& sh, uint64_t* bar, uint32_t parity,
                                              unsigned long long limit_ns, int* status) {
  const bool ok = wait_bar<PAIR>(sh, bar, parity, limit_ns, status);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Arrive on a barrier of the pair's rank-0 CTA (this CTA's own without a pair).
template <bool PAIR>
__device__ __forceinline__ void arrive_leader(const Shared& sh, uint64_t* bar) {
  if (PAIR) mbar_arrive_cluster(mapa_shared(smem_u32(bar), 0u));
  else mbar_arrive(smem_u32(bar));
}

// One 128-wide K chunk of a tile: four K = 32 steps, each an MMA per row
// block (gate and up, or two row blocks of W2) into its own accumulator, or,
// with a CTA pair, one M = 256 MMA over both CTAs' row blocks; `accum` turns
// on after the tile's first step.
template <bool PAIR, bool TWO>
__device__ __forceinline__ void issue_chunk(uint32_t d0, uint32_t d1, uint32_t a_lo, uint32_t b_lo, uint32_t sf,
                                            const uint32_t (&idesc)[4], uint32_t& accum) {
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
    if (PAIR) {
      // one M = 256 MMA: each CTA's own row block, its A scales at +0, the B
      // scales of all N columns at +8
      mma_mxf8f6f4_pair_lo(d0, a_lo + 2u * kb, b_lo + 2u * kb, kDescHiSw128, idesc[kb], sf + 0u, sf + 8u, accum);
    } else {
      mma_mxf8f6f4_lo(d0, a_lo + 2u * kb, b_lo + 2u * kb, kDescHiSw128, idesc[kb], sf + 0u, sf + 16u, accum);
      if (TWO)
        mma_mxf8f6f4_lo(d1, a_lo + (16384u >> 4) + 2u * kb, b_lo + 2u * kb, kDescHiSw128, idesc[kb], sf + 8u,
                        sf + 16u, accum);
    }
    accum = 1u;
  }
}

// The same K chunk (128 elements) with both operands packed E2M1: two K = 64
// steps per row block, each reading two scale bytes of the rows' TMEM words
// (sf_id 0, then 2); row block 2m + 1 starts 8 KB after block 2m.
template <bool TWO>
__device__ __forceinline__ void issue_chunk_a4(uint32_t d0, uint32_t d1, uint32_t a_lo, uint32_t b_lo, uint32_t sf,
                                               const uint32_t (&idesc)[2], uint32_t& accum) {
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    mma_mxf4_lo(d0, a_lo + 2u * kb, b_lo + 2u * kb, kDescHiSw64, idesc[kb], sf + 0u, sf + 16u, accum);
    if (TWO)
      mma_mxf4_lo(d1, a_lo + (8192u >> 4) + 2u * kb, b_lo + 2u * kb, kDescHiSw64, idesc[kb], sf + 8u, sf + 16u,
                  accum);
    accum = 1u;
  }
}

// PAIR: the kernel runs as clusters of two CTAs on neighbouring SMs.  A work
// unit is (expert, token tile, pair of weight tiles); rank r takes weight tile
// 2u + r of the unit's pair and half r of its token rows, and rank 0 issues
// M = 256 MMAs that use both CTAs' operands and write both CTAs' accumulators
// (the token rows each SM loads are halved against one CTA per tile).  The
// pipeline's full barriers and the accumulator-free barriers live in rank 0
// (rank 1's TMA loads, scale-staging and epilogue warps arrive on them
// remotely); the MMA commits free the stage and signal the accumulator in both
// CTAs at once.
// BT: the token-row scales are K-chunk-major (gathered rows, b_scales_t).
// EPI: 0 gate/up (SwiGLU + requantisation), 1 down (weighted combine), -1
// either (p.epi).  The wide schedule's launches take the specialised kernels
// (smaller code: 2% on the 8192-token layer).  The narrow schedule's two
// launches share one kernel (-1): the down launch's CTAs start as the gate/up
// CTAs leave, and with the gate/up launch's code still in the caches; with a
// kernel of its own the 16-token layer was 7 us slower (its code fetched cold).
// A4: MXFP4 activations (packed E2M1 operands, kind::mxf4): 1 yes, 0 no, -1
// either (p.a4).  The narrow schedule's kernels are specialised (the common
// MXFP8-activation kernel leaves the packed-FP4 code out: less code to fetch
// cold at the start of a small layer).
// The wide gate/up kernel (single CTA, gathered rows) runs 12 epilogue warps
// (three per lane quarter): its SwiGLU/requantisation epilogue drains the one
// accumulator buffer while the next tile's MMAs wait.
__host__ __device__ constexpr int epi_warps(bool pair, bool bt, int epi) { return (!pair && bt && epi == 0) ? 12 : 8; }
__host__ __device__ constexpr int gemm_threads(bool pair, bool bt, int epi) {
  return (kWarpEpi0 + epi_warps(pair, bt, epi)) * 32;
}

template <bool PAIR, bool BT, int EPI, int A4 = -1>
__global__ void __launch_bounds__(gemm_threads(PAIR, BT, EPI), 1)
    k_grouped_gemm(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_b) {
  constexpr int kEW = epi_warps(PAIR, BT, EPI);        // epilogue warps
  constexpr int kTh = gemm_threads(PAIR, BT, EPI);     // threads
  constexpr int kNH = kEW / 4;                         // epilogue warps per lane quarter
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.stages;

  Shared sh;
  sh.base = base;
  sh.offs = reinterpret_cast<int*>(base + p.off_meta);
  sh.prefix = sh.offs + (p.n_exp + 1);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + p.off_bar);
  sh.full = bars;
  sh.empty = bars + S;
  sh.acc_full = bars + 2 * S;
  sh.acc_empty = bars + 2 * S + 2;
  sh.drain = bars + 2 * S + 4;
  sh.exit_bar = bars + 2 * S + 5;
  sh.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 6);
  sh.abort_flag = reinterpret_cast<volatile int*>(bars + 2 * S + 7);
  sh.peer_full = bars + 2 * S + 8;                                 // S barriers
  sh.xfull = bars + 3 * S + 8;
  sh.xfree = bars + 3 * S + 9;
  sh.sf_cnt = reinterpret_cast<unsigned*>(bars + 3 * S + 10);      // S counters
  sh.rank = PAIR ? cluster_ctarank() : 0u;
  sh.hint_ns = p.hint_ns;
  const bool leader = sh.rank == 0;
  // work units: one per CTA, or one per CTA pair
  const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int unit_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  // ---- set-up that needs nothing from the previous grid (barriers, tensor
  // memory) runs before waiting on it; then the expert offsets, per-expert
  // tile counts and their prefix
  const int E1 = p.n_exp;  // experts of this launch
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      // a stage is full when its TMA bytes have landed (producer: 1 arrival
      // with the byte count) and the scale-staging warps have put its scale
      // factors into tensor memory (4 arrivals; with a pair, 1).  In a pair
      // each CTA's full barrier tracks its own copy of the stage, and rank 1
      // relays its completion to rank 0's peer_full barrier.
      mbar_init(smem_u32(&sh.full[s]), PAIR ? 2 : 5);
      mbar_init(smem_u32(&sh.empty[s]), 1);
      mbar_init(smem_u32(&sh.peer_full[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sh.acc_full[a]), 1);
      mbar_init(smem_u32(&sh.acc_empty[a]), PAIR ? 2 * kEW : kEW);
    }
    mbar_init(smem_u32(sh.drain), 1);
    mbar_init(smem_u32(sh.exit_bar), 1);
    mbar_init(smem_u32(sh.xfull), kEW);
    mbar_init(smem_u32(sh.xfree), kEW);
    for (int s = 0; s < S; ++s) sh.sf_cnt[s] = 0u;
    *sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(sh.tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(sh.tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  if (p.pdl == 1) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (p.pdl != 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = tid; i < E1 + 1; i += blockDim.x) sh.offs[i] = p.offsets[i];
  __syncthreads();
  // tile prefix: each thread owns a run of experts, warp 0..11 shuffle-scan
  {
    __shared__ int warp_tot[kTh / 32];
    const int per = (E1 + kTh - 1) / kTh;
    const int b0 = min(tid * per, E1), b1 = min(b0 + per, E1);
    int run = 0;
    for (int e = b0; e < b1; ++e) {
      const int cnt = sh.offs[e + 1] - sh.offs[e];
      run += p.MG * ((cnt + p.bn - 1) / p.bn);
    }
    int incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int acc = incl - run;
    for (int w = 0; w < warp; ++w) acc += warp_tot[w];
    for (int e = b0; e < b1; ++e) {
      sh.prefix[e] = acc;
      const int cnt = sh.offs[e + 1] - sh.offs[e];
      acc += p.MG * ((cnt + p.bn - 1) / p.bn);
    }
    if (b1 == E1 && b0 < b1) sh.prefix[E1] = acc;
    if (E1 == 0 && tid == 0) sh.prefix[0] = 0;
  }
  tc_fence_before();
  __syncthreads();
  // a pair's barriers must be initialised before the peer arrives on them
  if (PAIR) cluster_sync_all();
  tc_fence_after();
  const uint32_t tbase = *sh.tmem_slot;
  const int per_group = sh.prefix[E1];
  const int total = per_group * (p.NM / p.MG);
  const int NK = p.NK;

  if (warp == kWarpTma) {
    // ================================================================ producer
    // Lane 0 arms each stage and issues the weight-block TMA loads; the token
    // rows come either as one 2-D box of slot-ordered rows (the down GEMM's h,
    // or activation rows the wide schedule gathered into slot order first) or
    // as TMA gather4 loads of four token rows each, one per lane (the narrow
    // gate/up schedule: an expert's tokens are scattered over the activation
    // matrix).  The scale factors are staged by the scale warps.
    if (lane == 0) {
      prefetch_tensormap(&tm_a);
      prefetch_tensormap(&tm_b);
    }
    const bool gather = p.gather4 != 0;
    // ring position kept incrementally (no division by the runtime stage count)
    const uint32_t S_ = static_cast<uint32_t>(S);
    const int kps = p.kps;
    const unsigned long long lim = p.wait_limit_ns;
    int* const status = p.status;
    uint32_t it = 0, rs = 0, rph = 0;
    bool ok = true;
    bool b_ready = p.pdl != 2;  // mode 2: the B rows appear when the previous grid completes
    for (int t = unit0; t < total && ok; t += unit_step) {
      const Tile tl = decode_tile(t, sh, E1 - 1, p.MG, p.bn, per_group);
      // the tile's first prepared row block (a pair's CTA: its own block)
      const int blk_row = p.one ? tl.m : 2 * tl.m + (PAIR ? static_cast<int>(sh.rank) : 0);
      // a pair's MMA takes token rows [0, N/2) from rank 0 and [N/2, N) from
      // rank 1, N the tile's rows rounded up to 16
      int n_mma = (tl.rows + 15) & ~15;
      if (n_mma < 16) n_mma = 16;
      const int b_row0 = tl.p0 + (PAIR ? static_cast<int>(sh.rank) * (n_mma >> 1) : 0);
      // the tile's two row blocks are prepared blocks 2m and 2m + 1 of each K
      // chunk (gate and up block m in W1): one TMA box
      // gather: lane g loads rows 4g..4g+3 (padding rows repeat the last token).
      // The decode-size kernel reads their tokens once the tile's first weight
      // copy is on its way; the wide kernels (no gather) keep the read here,
      // out of their stage loop.
      const int n4 = gather ? (tl.rows + 3) / 4 : 0;
      int tok[4] = {0, 0, 0, 0};
      auto read_tok = [&]() {
        if (gather && lane < n4) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = min(4 * lane + j, tl.rows - 1);
            const int tt = __ldg(&p.sorted_slot[tl.p0 + r]) / (p.k + 1);
            if (tt < 0 || tt >= p.T) set_status(p.status, MX_ERR_DEVICE_ARG);
            tok[j] = (tt < 0 || tt >= p.T) ? 0 : tt;
          }
        }
      };
      if (EPI >= 0) read_tok();
      const uint32_t b_row = p.b_row;
      const int kx = (A4 < 0 ? p.a4 != 0 : A4 == 1) ? 64 : 128;  // bytes of a K chunk in a token row
      const uint32_t b_bytes = gather ? static_cast<uint32_t>(n4) * 4u * b_row : static_cast<uint32_t>(p.brows) * b_row;
      const uint32_t bytes = ((PAIR || p.one ? 1u : 2u) * p.a_tx + b_bytes) * static_cast<uint32_t>(kps);
      for (int ks = 0; ks < NK; ks += kps) {
        const uint32_t s = rs, ph = rph;
        if (!warp_wait_bar<PAIR>(sh, &sh.empty[s], ph ^ 1u, lim, status)) {
          ok = false;
          break;
        }
        const uint32_t full = smem_u32(&sh.full[s]);
        const uint32_t su = s * static_cast<uint32_t>(kps);  // first chunk slot
        if (lane == 0) {
          mbar_arrive_expect_tx(full, bytes);
          // the stage's weight blocks in one copy: row blocks 2m and 2m + 1 (one
          // with a pair; a block past the last row block is filled with zeros and
          // still counted) of its kps K chunks, chunk-major in shared memory.
          // Fewer, larger copies: a TMA copy has a fixed cost of its own, and a
          // stage of MXFP4 blocks is only 8 KB per block.
          uint8_t* a_s = base + p.off_a + su * p.a_slot;
          tma_load_4d(smem_u32(a_s), &tm_a, 0, 0, blk_row, (tl.e + p.e_base) * NK + ks, full);
        }
        if (EPI < 0 && ks == 0) read_tok();
        if (!b_ready) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          b_ready = true;
        }
        for (int u = 0; u < kps; ++u) {
          const int kc = ks + u;
          const uint32_t b_s = smem_u32(base + p.off_b + (su + u) * p.brows * b_row);
          if (lane == 0 && !gather) tma_load_2d(b_s, &tm_b, kc * kx, b_row0, full);
          __syncwarp();
          if (gather && lane < n4)
            tma_gather4(b_s + static_cast<uint32_t>(lane) * 4u * b_row, &tm_b, kc * kx, tok[0], tok[1], tok[2],
                        tok[3], full);
        }
        ++it;  // fills armed
        if (++rs == S_) {
          rs = 0;
          rph ^= 1u;
        }
      }
    }
    // drain: every fill this warp armed has landed before the CTA exits
    if (lane == 0) {
      const uint32_t n_fills = it;
      for (int s = 0; s < S && static_cast<uint32_t>(s) < n_fills; ++s) {
        const uint32_t last = n_fills - 1 - ((n_fills - 1 - s) % S);
        mbar_wait(smem_u32(&sh.full[s]), (last / S) & 1u, 100000000ull);
      }
    }
  } else if (PAIR && warp == kWarpMma && !leader) {
    // ================================================================ pair relay
    // Rank 1 (whose MMA warp issues nothing): once its copy of a stage is full
    // (its TMA bytes landed, its scale factors stored), tell rank 0, whose
    // MMAs read both copies.
    if (lane == 0) {
      const uint32_t S_ = static_cast<uint32_t>(S);
      const int NKs = NK / p.kps;
      uint32_t rs = 0, rph = 0;
      bool ok = true;
      for (int t = unit0; t < total && ok; t += unit_step) {
        for (int ks = 0; ks < NKs; ++ks) {
          const uint32_t s = rs, ph = rph;
          if (++rs == S_) {
            rs = 0;
            rph ^= 1u;
          }
          if (!wait_bar<PAIR, false>(sh, &sh.full[s], ph, p.wait_limit_ns, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(mapa_shared(smem_u32(&sh.peer_full[s]), 0u));
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ================================================================ MMA issuer
    if (lane == 0 && (!PAIR || leader)) {
      // everything the issue loop needs lives in registers, and the ring and
      // accumulator positions advance incrementally: the single issuing thread's
      // per-stage latency (divisions, parameter reloads) is MMA issue time lost
      const uint32_t S_ = static_cast<uint32_t>(S);
      const uint32_t acc_bufs = static_cast<uint32_t>(p.acc_bufs);
      const unsigned long long lim = p.wait_limit_ns;
      int* const status = p.status;
      const int NKs = NK / p.kps;  // stages per tile
      uint32_t rs = 0, rph = 0, ab = 0, aph = 0;
      const uint32_t afmt = p.afmt == MX_E4M3 ? kFmtE4M3 : kFmtE2M1;
      const uint32_t sf_base = tbase + p.sf_col0;
      const uint32_t a_base = smem_u32(base + p.off_a);
      const uint32_t b_base = smem_u32(base + p.off_b);
      const uint32_t b_stride16 = (static_cast<uint32_t>(p.brows) * p.b_row) >> 4;
      const uint32_t a16 = p.a_slot >> 4;  // A chunk slot stride in 16-byte units
      const bool a4 = A4 < 0 ? p.a4 != 0 : A4 == 1;
      const uint32_t kps = static_cast<uint32_t>(p.kps);
      // descriptors of slot 0 (start address field is addr >> 4; slots add to it)
      const uint32_t a_lo0 = desc_lo_sw128(a_base);
      const uint32_t b_lo0 = desc_lo_sw128(b_base);
      constexpr uint32_t kM = PAIR ? 256u : 128u;
      bool ok = true;
      for (int t = unit0; t < total && ok; t += unit_step) {
        const Tile tl = decode_tile(t, sh, E1 - 1, p.MG, p.bn, per_group);
        const bool two = !PAIR && !p.one && (EPI == 0 || (EPI < 0 && p.epi == 0) || (2 * tl.m + 1 < p.RB));
        uint32_t n_mma = static_cast<uint32_t>((tl.rows + 15) & ~15);
        if (n_mma < 16) n_mma = 16;
        if (!wait_bar<PAIR>(sh, &sh.acc_empty[ab], aph ^ 1u, lim, status)) break;
        tc_fence_after();
        const uint32_t d0 = tbase + ab * p.acc_cols;
        const uint32_t d1 = d0 + static_cast<uint32_t>(p.bn);
        uint32_t idesc[4], idesc4[2];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) idesc[kb] = idesc_mx(afmt, kFmtE4M3, kM, n_mma, kb, kb);
        idesc4[0] = idesc_mxf4(kM, n_mma, 0);
        idesc4[1] = idesc_mxf4(kM, n_mma, 2);
        uint32_t accum = 0u;
        for (int ks = 0; ks < NKs; ++ks) {
          const uint32_t s = rs, ph = rph;
          if (++rs == S_) {
            rs = 0;
            rph ^= 1u;
          }
          if (!wait_bar<PAIR, false>(sh, &sh.full[s], ph, lim, status) ||
              (PAIR && !wait_bar<PAIR, false>(sh, &sh.peer_full[s], ph, lim, status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // all the stage's MMAs back to back (its scale factors are already in
          // tensor memory): the single issuing thread's work between two MMAs
          // is tensor time
          const uint32_t slot0 = s * kps;
          constexpr uint32_t sfc = PAIR ? kSfColsPerChunkPair : kSfColsPerChunk;
          if (!PAIR && a4) {
            for (uint32_t u = 0; u < kps; ++u) {
              const uint32_t al = a_lo0 + (slot0 + u) * a16, bl = b_lo0 + (slot0 + u) * b_stride16;
              const uint32_t sf = sf_base + (slot0 + u) * sfc;
              if (two) issue_chunk_a4<true>(d0, d1, al, bl, sf, idesc4, accum);
              else issue_chunk_a4<false>(d0, d1, al, bl, sf, idesc4, accum);
            }
          } else if (two) {
            issue_chunk<PAIR, true>(d0, d1, a_lo0 + slot0 * a16, b_lo0 + slot0 * b_stride16, sf_base + slot0 * sfc,
                                    idesc, accum);
            if (kps == 2)
              issue_chunk<PAIR, true>(d0, d1, a_lo0 + (slot0 + 1) * a16, b_lo0 + (slot0 + 1) * b_stride16,
                                      sf_base + (slot0 + 1) * sfc, idesc, accum);
          } else {
            issue_chunk<PAIR, false>(d0, d1, a_lo0 + slot0 * a16, b_lo0 + slot0 * b_stride16, sf_base + slot0 * sfc,
                                     idesc, accum);
            if (kps == 2)
              issue_chunk<PAIR, false>(d0, d1, a_lo0 + (slot0 + 1) * a16, b_lo0 + (slot0 + 1) * b_stride16,
                                       sf_base + (slot0 + 1) * sfc, idesc, accum);
          }
          if (PAIR) mma_commit_pair(smem_u32(&sh.empty[s]), 3);
          else mma_commit(smem_u32(&sh.empty[s]));
        }
        if (!ok) break;
        if (PAIR) mma_commit_pair(smem_u32(&sh.acc_full[ab]), 3);
        else mma_commit(smem_u32(&sh.acc_full[ab]));
        if (++ab == acc_bufs) {
          ab = 0;
          aph ^= 1u;
        }
      }
      // every MMA this thread issued has completed before TMEM is released
      if (PAIR) mma_commit_pair(smem_u32(sh.drain), 1);
      else mma_commit(smem_u32(sh.drain));
      mbar_wait(smem_u32(sh.drain), 0, 100000000ull);
    }
  } else if (warp >= kWarpSf0 && warp < kWarpSf0 + 4) {
    // ================================================================ scale staging
    // Per stage: the weight (A) scale blocks of the tile's two row blocks (one
    // 16-byte word per lane and block, already in the tensor-memory order) and
    // the token-row (B) scales (one 32-bit word per row and chunk, all N rows
    // of the tile also with a pair) are read from global memory two K chunks
    // ahead of the chunk being stored (three register buffers: a chunk's loads
    // are in flight while earlier chunks wait for their slot and are stored),
    // then stored with tcgen05.st into this warp's TMEM lane quarter
    // (all four quarters hold the same words, the layout the block-scaled MMA
    // reads).  Then the stage's full barrier gets its arrival: one per warp,
    // or, with a pair, one for all four warps from the last of them to finish.
    struct ScaleBuf {  // one K chunk
      uint32_t bw[8];
      uint4 a0, a1;
    };
    const int q = warp & 3;
    const int K32 = p.K / 32;
    const uint32_t S_ = static_cast<uint32_t>(S);
    const int kps = p.kps, bn = p.bn;
    const unsigned long long lim = p.wait_limit_ns;
    int* const status = p.status;
    const uint32_t col0 = tbase + (static_cast<uint32_t>(32 * q) << 16) + p.sf_col0;
    const uint4* const wsc = reinterpret_cast<const uint4*>(p.w_scales);
    // token-row scales: by row ([rows][K/128] words, the word of chunk kc at
    // +kc), or K-chunk-major for gathered rows ([K/128][n_rows], at +kc n_rows:
    // a chunk's words of consecutive rows are adjacent, one coalesced load)
    const uint32_t* const bsc = BT ? p.b_scales_t : reinterpret_cast<const uint32_t*>(p.b_scales);
    uint32_t rs = 0, rph = 0;
    bool ok = true;
    if (p.pdl == 2) asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int t = unit0; t < total && ok; t += unit_step) {
      const Tile tl = decode_tile(t, sh, E1 - 1, p.MG, p.bn, per_group);
      // the tile's first prepared row block (a pair's CTA: its own, the only one)
      const int blk_row = p.one ? tl.m : 2 * tl.m + (PAIR ? static_cast<int>(sh.rank) : 0);
      const bool two = !PAIR && !p.one && 2 * tl.m + 1 < p.RB;
      // warm L2 with the tile's weight-scale blocks (128-byte lines, 4 per
      // block, one or two blocks per chunk): the per-stage loads below then hit
      // L2 instead of waiting on DRAM.  Kernels that run the gate/up epilogue
      // issue them before reading the tile's tokens from the permutation (a
      // dependent load); the down-only kernel after its row offsets.
      auto prefetch_wsc = [&]() {
        const int lines = two ? 8 : 4;
        const int sft = tid - kWarpSf0 * 32;
        for (int i = sft; i < NK * lines; i += 128) {
          const int kc = i / lines, line = i - kc * lines;
          const uint4* blk = wsc + static_cast<size_t>(((tl.e + p.e_base) * NK + kc) * p.RB + blk_row) * 32;
          prefetch_l2(reinterpret_cast<const uint8_t*>(blk) + line * 128);
        }
      };
      if (EPI != 1) prefetch_wsc();
      // rows 32j + lane of this tile: the word offset of their scale rows
      // (-1: a padding row)
      int roww[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = 32 * j + lane;
        roww[j] = -1;
        if (BT && r < tl.rows) {
          roww[j] = tl.p0 + r;
        } else if (!BT && r < tl.rows) {
          int src_row = tl.p0 + r;
          if (EPI == 0 || (EPI < 0 && p.epi == 0)) {
            src_row = __ldg(&p.sorted_slot[tl.p0 + r]) / (p.k + 1);
            if (src_row < 0 || src_row >= p.T) {
              set_status(status, MX_ERR_DEVICE_ARG);
              src_row = 0;
            }
          }
          roww[j] = src_row * (K32 / 4);
        }
      }
      if (EPI == 1) prefetch_wsc();
      auto load = [&](ScaleBuf& b, int kc) {
        if (BT) {
          const uint32_t* const bk = bsc + static_cast<size_t>(kc) * static_cast<size_t>(p.n_rows);
#pragma unroll
          for (int j = 0; j < 8; ++j) b.bw[j] = roww[j] >= 0 ? __ldg(bk + roww[j]) : 0x7F7F7F7Fu;
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) b.bw[j] = roww[j] >= 0 ? __ldg(bsc + roww[j] + kc) : 0x7F7F7F7Fu;
        }
        const uint4* blk = wsc + static_cast<size_t>(((tl.e + p.e_base) * NK + kc) * p.RB + blk_row) * 32;
        b.a0 = __ldg(blk + lane);
        b.a1 = two ? __ldg(blk + 32 + lane) : make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      };
      // store chunk kc from `cur` (its loads issued two chunks earlier) after
      // issuing the loads of chunk kc + 2 into `nxt`; the stage's slot is
      // awaited at its first chunk and its arrival made after its last
      uint32_t s = 0;
      auto step = [&](ScaleBuf& cur, ScaleBuf& nxt, int kc) {
        if (kc + 2 < NK) load(nxt, kc + 2);
        const int u = kc % kps;
        if (u == 0) {
          s = rs;
          const uint32_t ph = rph;
          if (++rs == S_) {
            rs = 0;
            rph ^= 1u;
          }
          if (!warp_wait_bar<PAIR>(sh, &sh.empty[s], ph ^ 1u, lim, status)) return false;
        }
        // chunk slot: A scales of row block 2m at +0, of 2m + 1 at +8, B at
        // +16 (column j of a block holds rows 32j + lane; B: j < 8, N <= 256);
        // a pair's CTA: its one A block at +0, B at +8
        constexpr uint32_t sfc = PAIR ? kSfColsPerChunkPair : kSfColsPerChunk;
        constexpr uint32_t b_col = PAIR ? 8u : 16u;
        const uint32_t col = col0 + (s * static_cast<uint32_t>(kps) + static_cast<uint32_t>(u)) * sfc;
        __syncwarp();
        tmem_st_32x32b_x4(col + 0u, cur.a0.x, cur.a0.y, cur.a0.z, cur.a0.w);
        if (!PAIR) tmem_st_32x32b_x4(col + 8u, cur.a1.x, cur.a1.y, cur.a1.z, cur.a1.w);
        if (bn > 128) tmem_st_32x32b_x8(col + b_col, cur.bw);
        else tmem_st_32x32b_x4(col + b_col, cur.bw[0], cur.bw[1], cur.bw[2], cur.bw[3]);
        if (u != kps - 1) return true;
        tmem_st_wait();
        tc_fence_before();
        if (PAIR) {
          // the last of the four scale warps to finish this stage (a shared
          // counter per slot, reset by that warp; nothing blocks) arrives for all
          __syncwarp();
          if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&sh.sf_cnt[s], 1u) == 3u) {
              __threadfence_block();
              sh.sf_cnt[s] = 0u;
              mbar_arrive(smem_u32(&sh.full[s]));
            }
          }
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sh.full[s]));
        }
        return true;
      };
      ScaleBuf b0, b1, b2;
      load(b0, 0);
      if (NK > 1) load(b1, 1);
      for (int kc = 0; kc < NK; kc += 3) {
        if (!step(b0, b2, kc)) {
          ok = false;
          break;
        }
        if (kc + 1 >= NK) break;
        if (!step(b1, b0, kc + 1)) {
          ok = false;
          break;
        }
        if (kc + 2 >= NK) break;
        if (!step(b2, b1, kc + 2)) {
          ok = false;
          break;
        }
      }
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kEW) {
    // ================================================================ epilogue
    const int q = warp & 3;                   // TMEM lane quarter of this warp
    const int half = (warp - kWarpEpi0) >> 2;  // which alternate column chunks (of kNH)
    uint8_t* const ebuf =
        base + p.off_epi + static_cast<uint32_t>(warp - kWarpEpi0) * epi_buf_bytes(EPI < 0 ? p.epi : EPI);
    const uint32_t acc_bufs = static_cast<uint32_t>(p.acc_bufs);
    uint32_t ab = 0, aph = 0, ab_next = 0, aph_next = 0;
    uint32_t xph = 0;  // pair gate/up: phase of the exchange barriers
    for (int t = unit0; t < total; t += unit_step) {
      const Tile tl = decode_tile(t, sh, E1 - 1, p.MG, p.bn, per_group);
      ab = ab_next;
      aph = aph_next;
      if (++ab_next == acc_bufs) {
        ab_next = 0;
        aph_next ^= 1u;
      }
      if (!warp_wait_bar<PAIR>(sh, &sh.acc_full[ab], aph, p.wait_limit_ns, p.status)) break;
      tc_fence_after();
      __syncwarp();
      const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
      const uint32_t d0 = tbase + lane_base + ab * p.acc_cols;
      const uint32_t d1 = d0 + static_cast<uint32_t>(p.bn);
      if (EPI == 0 || (EPI < 0 && p.epi == 0)) {
        const int i0 = tl.m * 128 + 32 * q;  // this warp's 32 rows of I (one MX block of h)
        const int I = p.I, I32 = p.I / 32;
        uint8_t* const h_codes = p.h_codes;
        uint8_t* const h_scales = p.h_scales;
        const bool act_oai = p.act != 0;
        const float alpha = p.alpha, limit = p.limit;
        const bool h4 = A4 < 0 ? p.a4 != 0 : A4 == 1;  // h re-quantised to MXFP4 (packed E2M1, I/2 bytes a row)
        // 8 columns at a time, each step over all 8 so that the per-column
        // chains (SwiGLU, warp amax, exponent, encode) overlap; the tensor-
        // memory loads of the warp's next 8 columns are in flight while the
        // current ones are processed (two register sets, computed in place)
        auto process = [&](uint32_t (&g)[8], uint32_t (&u)[8], int c0) {
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            // silu(g) * u with the fast reciprocal: h is re-quantised to 3
            // mantissa bits right after, far coarser than its 2-ulp error.
            // SwiGLU-OAI: the gate clamped above at `limit`, the up projection
            // to [-limit, limit], h = g * sigmoid(alpha * g) * (u + 1).
            float gv = __uint_as_float(g[cc]);
            float uv = __uint_as_float(u[cc]);
            float sl = 1.0f;
            if (act_oai) {
              gv = fminf(gv, limit);
              uv = fminf(fmaxf(uv, -limit), limit) + 1.0f;
              sl = alpha;
            }
            const float hv = __fdividef(gv, 1.0f + __expf(-sl * gv)) * uv;
            g[cc] = __float_as_uint(hv);
            u[cc] = __float_as_uint(hv) & 0x7FFFFFFFu;
          }
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) u[cc] = __reduce_max_sync(0xffffffffu, u[cc]);
          if (h4) {
            // MXFP4: lanes 2i and 2i + 1 (rows 2i, 2i + 1 of I) share one byte,
            // row 2i in the low nibble; per column 16 bytes through the
            // per-warp tile [8 columns][16 bytes]
            int my_s4 = 0;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
              const int sc = mx_block_exponent(u[cc], 2);
              const uint32_t code = enc_e2m1(__uint_as_float(g[cc]) * pow2_neg(sc));
              const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
              if ((lane & 1) == 0) ebuf[cc * 16 + (lane >> 1)] = static_cast<uint8_t>(code | (hi << 4));
              if (lane == cc) my_s4 = sc;
            }
            __syncwarp();
            const int nv = tl.rows - c0;
            if (lane < 8 && lane < nv) {
              const uint4 v = *reinterpret_cast<const uint4*>(ebuf + lane * 16);
              *reinterpret_cast<uint4*>(h_codes + static_cast<size_t>(tl.p0 + c0 + lane) * (I / 2) + i0 / 2) = v;
              h_scales[static_cast<size_t>(tl.p0 + c0 + lane) * I32 + i0 / 32] = static_cast<uint8_t>(my_s4 + 127);
            }
            __syncwarp();
            return;
          }
          // codes go through a per-warp shared-memory tile [8 columns][32 rows
          // of I] so that each lane writes one 16-byte run of an h row (byte
          // stores from every lane, one per column, throttle the store path)
          int my_s = 0;  // lane j < 8: the scale of column j
#pragma unroll
          for (int cc = 0; cc < 8; cc += 2) {
            const int s0 = mx_block_exponent(u[cc], 8);
            const int s1 = mx_block_exponent(u[cc + 1], 8);
            const uint32_t codes =
                enc_e4m3x2(__uint_as_float(g[cc]) * pow2_neg(s0), __uint_as_float(g[cc + 1]) * pow2_neg(s1));
            ebuf[cc * 32 + lane] = static_cast<uint8_t>(codes);
            ebuf[(cc + 1) * 32 + lane] = static_cast<uint8_t>(codes >> 8);
            if (lane == cc) my_s = s0;
            if (lane == cc + 1) my_s = s1;
          }
          __syncwarp();
          const int nvalid = tl.rows - c0;
          const int col = lane >> 1;
          if (lane < 16) {
            const uint4 v = *reinterpret_cast<const uint4*>(ebuf + col * 32 + (lane & 1) * 16);
            if (col < nvalid)
              *reinterpret_cast<uint4*>(h_codes + static_cast<size_t>(tl.p0 + c0 + col) * I + i0 + (lane & 1) * 16) = v;
          }
          if (lane < 8 && lane < nvalid)
            h_scales[static_cast<size_t>(tl.p0 + c0 + lane) * I32 + i0 / 32] = static_cast<uint8_t>(my_s + 127);
          __syncwarp();
        };
        if (PAIR) {
          // rank 0 holds g (gate block m), rank 1 u (up block m), for all N
          // tokens of the tile; rank 0 finishes tokens [0, N/2), rank 1
          // [N/2, N), each after receiving the other's values for its half in
          // its exchange buffer (rows of I x its tokens, row stride xs words)
          int nmma = (tl.rows + 15) & ~15;
          if (nmma < 16) nmma = 16;
          const int hw = nmma >> 1;
          const int own0 = static_cast<int>(sh.rank) * hw, oth0 = hw - own0;
          const uint32_t xs = p.xs;
          float* const xmine = reinterpret_cast<float*>(base + p.off_x);
          const uint32_t xpeer = mapa_shared(smem_u32(xmine), sh.rank ^ 1u);
          const uint32_t row = static_cast<uint32_t>(32 * q + lane);
          // the partner has read its buffer for the previous tile
          if (!warp_wait_bar<PAIR>(sh, sh.xfree, xph ^ 1u, p.wait_limit_ns, p.status)) break;
          for (int c0 = oth0 + 8 * half; c0 < oth0 + hw && c0 < tl.rows; c0 += 16) {
            uint32_t v[8];
            __syncwarp();
            tmem_ld_32x32b_x8(d0 + c0, v);
            tmem_ld_wait();
            const uint32_t a = xpeer + (row * xs + static_cast<uint32_t>(c0 - oth0)) * 4u;
            st_shared_cluster_v4(a, v[0], v[1], v[2], v[3]);
            st_shared_cluster_v4(a + 16u, v[4], v[5], v[6], v[7]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(sh.xfull), sh.rank ^ 1u));
          // the partner's values for this CTA's tokens have arrived
          if (!warp_wait_bar<PAIR>(sh, sh.xfull, xph, p.wait_limit_ns, p.status)) break;
          for (int c0 = own0 + 8 * half; c0 < own0 + hw && c0 < tl.rows; c0 += 16) {
            uint32_t mine[8], other[8];
            __syncwarp();
            tmem_ld_32x32b_x8(d0 + c0, mine);
            const uint4* xp = reinterpret_cast<const uint4*>(xmine + row * xs + static_cast<uint32_t>(c0 - own0));
            const uint4 o0 = xp[0], o1 = xp[1];
            other[0] = o0.x, other[1] = o0.y, other[2] = o0.z, other[3] = o0.w;
            other[4] = o1.x, other[5] = o1.y, other[6] = o1.z, other[7] = o1.w;
            tmem_ld_wait();
            if (sh.rank == 0) process(mine, other, c0);
            else process(other, mine, c0);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(sh.xfree), sh.rank ^ 1u));
          xph ^= 1u;
        } else {
        uint32_t ga[8], ua[8], gb[8], ub[8];
        int c0 = 8 * half;  // 8-column chunks dealt round-robin to the quarter's kNH warps
        if (c0 < tl.rows) {
          __syncwarp();
          tmem_ld_32x32b_x8(d0 + c0, ga);
          tmem_ld_32x32b_x8(d1 + c0, ua);
          tmem_ld_wait();
        }
        while (c0 < tl.rows) {
          const int c1 = c0 + 8 * kNH;
          if (c1 < tl.rows) {
            tmem_ld_32x32b_x8(d0 + c1, gb);
            tmem_ld_32x32b_x8(d1 + c1, ub);
          }
          process(ga, ua, c0);
          if (c1 >= tl.rows) break;
          tmem_ld_wait();
          const int c2 = c1 + 8 * kNH;
          if (c2 < tl.rows) {
            tmem_ld_32x32b_x8(d0 + c2, ga);
            tmem_ld_32x32b_x8(d1 + c2, ua);
          }
          process(gb, ub, c1);
          if (c2 >= tl.rows) break;
          tmem_ld_wait();
          c0 = c2;
        }
        }
      } else {
        // W2 row blocks 2m and 2m + 1 (a pair's CTA: its own one; one block a tile: m)
        const int blk_row = p.one ? tl.m : 2 * tl.m + (PAIR ? static_cast<int>(sh.rank) : 0);
        const bool two = !PAIR && !p.one && 2 * tl.m + 1 < p.RB;
        float* const out = p.out;
        const int H = p.H;
        float* const ebf = reinterpret_cast<float*>(ebuf);
        for (int c0 = 32 * half; c0 < tl.rows; c0 += 32 * kNH) {
          // lane n: token and combine weight of column c0 + n
          int tok = 0;
          float wt = 0.0f;
          if (c0 + lane < tl.rows) {
            const int slot = __ldg(&p.sorted_slot[tl.p0 + c0 + lane]);
            const int tt = slot / (p.k + 1), j = slot - tt * (p.k + 1);
            if (tt >= 0 && tt < p.T) {
              tok = tt;
              wt = j == p.k ? 1.0f : __ldg(&p.topk_w[static_cast<size_t>(tt) * p.k + j]);
            } else {
              set_status(p.status, MX_ERR_DEVICE_ARG);
            }
          }
          for (int sub = 0; sub < (two ? 2 : 1); ++sub) {
            // both 16-column halves of this row block's 32 columns in flight at
            // once, then one wait
            const uint32_t d = sub == 0 ? d0 : d1;
            uint32_t a[2][16];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              if (c0 + 16 * hh < tl.rows) tmem_ld_32x32b_x16(d + c0 + 16 * hh, a[hh]);
            tmem_ld_wait();
            const int o0 = (blk_row + sub) * 128 + 32 * q;  // this warp's 32 rows of H
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int h0 = 16 * hh;
              if (c0 + h0 >= tl.rows) break;
              // weighted values through the per-warp transpose tile [8 columns]
              // [32 rows of H], then four consecutive H values per lane and
              // column: one 16-byte vector reduction instead of four scalar ones
#pragma unroll
              for (int c8 = 0; c8 < 16; c8 += 8) {
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                  ebf[cc * 32 + lane] = __shfl_sync(0xffffffffu, wt, h0 + c8 + cc) * __uint_as_float(a[hh][c8 + cc]);
                __syncwarp();
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                  const int col = c8 + 4 * r + (lane >> 3);
                  const int tn = __shfl_sync(0xffffffffu, tok, h0 + col);
                  const float4 v = *reinterpret_cast<const float4*>(ebf + (col - c8) * 32 + (lane & 7) * 4);
                  if (c0 + h0 + col < tl.rows)
                    red_add_v4(out + static_cast<size_t>(tn) * H + o0 + (lane & 7) * 4, v);
                }
                __syncwarp();
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader<PAIR>(sh, &sh.acc_empty[ab]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) {
    // neither CTA of the pair leaves (or frees tensor memory, which is
    // allocated and freed by both at once) while the other can still arrive
    // on its barriers, load into its shared memory or be written by its MMAs:
    // each tells the other that all its roles are done (rank 0's MMAs have
    // drained by then) and waits for the same word from the other
    if (tid == 0) {
      mbar_arrive_cluster(mapa_shared(smem_u32(sh.exit_bar), sh.rank ^ 1u));
      const uint64_t t0 = globaltimer_ns();
      const unsigned long long lim = 8ull * p.wait_limit_ns + 100000000ull;
      while (!mbar_try_wait_cluster_sleep(smem_u32(sh.exit_bar), 0u, 20000u)) {
        if (globaltimer_ns() - t0 > lim) {
          set_status(p.status, MX_ERR_TIMEOUT);
          break;
        }
      }
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == kWarpMma) {
    __syncwarp();
    if (PAIR) tmem_dealloc_pair(tbase, kTmemCols);
    else tmem_dealloc(tbase, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

static int sm_count_gemm() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 152;
  }
  return n;
}

// Transaction bytes one weight-block TMA adds to its mbarrier: the bytes read
// from global memory (MXFP4 blocks are 8 KB packed, 16 KB once unpacked into
// shared memory).
static uint32_t weight_block_tx_bytes(int fmt) { return fmt == MX_E4M3 ? 16384u : 8192u; }

bool pair_supported(const GemmArgs& a) {
  // each CTA of a pair takes one row block of every weight tile (so every
  // tile needs both), with token rows in slot order (2-D boxes) split in halves
  const int rows = a.epi == 0 ? 2 * a.I : a.H;
  return !a.gather4 && !a.a4 && (rows / 128) % 2 == 0 && a.bn % 32 == 0 && a.bn >= 32 && a.bn <= 256;
}

// ---- optional per-launch timing (mx_debug_time_gemms)
namespace {
constexpr int kMaxTimed = 4096;
struct GemmTimer {
  std::mutex m;
  bool on = false;
  int dev = -1;  // device of the events (set at the first recorded launch)
  int n = 0;
  cudaEvent_t ev[kMaxTimed][2] = {};
  int epi[kMaxTimed] = {};
};
GemmTimer& gemm_timer() {
  static GemmTimer t;
  return t;
}
// the slot to record this launch into (-1: not timing, full or another device)
int timer_begin(int epi, cudaStream_t s) {
  GemmTimer& t = gemm_timer();
  std::lock_guard<std::mutex> g(t.m);
  if (!t.on || t.n >= kMaxTimed) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (t.dev < 0) t.dev = dev;
  if (dev != t.dev) return -1;
  const int i = t.n;
  for (int j = 0; j < 2; ++j)
    if (!t.ev[i][j] && cudaEventCreate(&t.ev[i][j]) != cudaSuccess) return -1;
  if (cudaEventRecord(t.ev[i][0], s) != cudaSuccess) return -1;
  t.epi[i] = epi;
  ++t.n;
  return i;
}
void timer_end(int i, cudaStream_t s) {
  if (i < 0) return;
  GemmTimer& t = gemm_timer();
  std::lock_guard<std::mutex> g(t.m);
  cudaEventRecord(t.ev[i][1], s);
}
}  // namespace

void gemm_timing_enable(bool on) {
  GemmTimer& t = gemm_timer();
  std::lock_guard<std::mutex> g(t.m);
  t.on = on;
  t.n = 0;
}

int gemm_timing_read(float* ms, int* epi, int max) {
  GemmTimer& t = gemm_timer();
  std::lock_guard<std::mutex> g(t.m);
  const int n = t.n;
  int rc = n;
  for (int i = 0; i < n && i < max; ++i) {
    float v = 0.f;
    if (cudaEventSynchronize(t.ev[i][1]) != cudaSuccess || cudaEventElapsedTime(&v, t.ev[i][0], t.ev[i][1]) != cudaSuccess)
      rc = -1;
    if (ms) ms[i] = v;
    if (epi) epi[i] = t.epi[i];
  }
  t.n = 0;
  return rc;
}

cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t stream) {
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  const bool pair = a.pair != 0;
  if (pair && !pair_supported(a)) return cudaErrorInvalidConfiguration;
  GemmParams p{};
  p.epi = a.epi;
  p.afmt = a.fmt;
  p.T = a.T;
  p.H = a.H;
  p.I = a.I;
  p.E = a.E;
  p.k = a.k;
  p.n_exp = a.n_exp > 0 ? a.n_exp : a.E + 1;
  p.e_base = a.e_base;
  p.act = a.act;
  p.alpha = a.alpha;
  p.limit = a.limit;
  const int rows = a.epi == 0 ? 2 * a.I : a.H;
  p.K = a.epi == 0 ? a.H : a.I;
  p.NK = p.K / 128;
  p.RB = rows / 128;
  // weight tiles of two row blocks (gate and up block m, or W2 blocks 2m and
  // 2m + 1); a CTA pair splits each tile's two blocks between its CTAs
  // one row block per tile: the down GEMM on wide token tiles (MXFP8 operands)
  p.one = (a.epi == 1 && !pair && !a.a4 && a.one_blk) ? 1 : 0;
  p.NM = a.epi == 0 ? a.I / 128 : p.one ? p.RB : (p.RB + 1) / 2;
  // down GEMM: split the weight tiles into groups so that one group's slice of
  // `out` (T rows x the group's 256-column blocks, fp32) stays within ~16 MB of
  // L2 while every expert's atomic combine lands on it
  p.MG = p.NM;
  if (a.epi == 1) {
    int groups = 1;
    const double out_bytes = 4.0 * a.T * a.H;
    while (out_bytes / groups > 16.0 * 1024 * 1024 && p.NM % (groups * 2) == 0) groups *= 2;
    if (const char* env = std::getenv("MXMOE_MGROUPS")) {
      const int v = std::atoi(env);
      if (v >= 1 && p.NM % v == 0) groups = v;
    }
    p.MG = p.NM / groups;
  }
  p.bn = a.bn;
  p.brows = pair ? a.bn / 2 : a.bn;
  p.sfc = pair ? kSfColsPerChunkPair : kSfColsPerChunk;
  p.acc_cols = (pair || p.one ? 1u : 2u) * static_cast<uint32_t>(a.bn);
  p.xs = static_cast<uint32_t>(a.bn / 2 + 4);
  p.n_rows = a.n_rows;
  p.a_tx = weight_block_tx_bytes(a.fmt);
  const PreparedLayout L = prepared_layout(a.E + 1, rows, p.K, a.fmt, a.epi == 0 ? 1 : 0);
  p.w_scales = static_cast<const uint8_t*>(a.w_prep) + L.scales_offset;
  p.b_scales = a.b_scales;
  p.b_scales_t = a.b_scales_t;
  p.offsets = a.offsets;
  p.sorted_slot = a.sorted_slot;
  p.topk_w = a.topk_w;
  p.h_codes = a.h_codes;
  p.h_scales = a.h_scales;
  p.out = a.out;
  p.status = a.status;
  p.wait_limit_ns = a.wait_limit_ns;
  p.gather4 = a.gather4;
  p.pdl = a.pdl;
  p.hint_ns = 20000u;
  if (const char* env = std::getenv("MXMOE_PAIR_HINT_NS")) p.hint_ns = static_cast<uint32_t>(std::atoi(env));
  // packed E2M1 operands: weight blocks of 8 KB (64-byte rows) and token rows
  // of 64 bytes per K chunk stay packed in shared memory (64-byte swizzle)
  p.a4 = a.a4;
  p.a_slot = (pair || p.one) ? 16384u : a.a4 ? 16384u : 32768u;
  p.b_row = a.a4 ? 64u : 128u;

  // shared memory and tensor memory plan for `kps` 128-wide K chunks per
  // pipeline stage: returns the stage count (0 if fewer than two fit)
  const uint32_t meta_bytes = (static_cast<uint32_t>(p.n_exp + 1) * 8u + 127u) & ~127u;
  int dev = 0;
  cudaGetDevice(&dev);
  int max_smem = 0;
  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const int n_epi_warps = epi_warps(pair, a.b_scales_t != nullptr, a.epi);
  const uint32_t epi_bytes = static_cast<uint32_t>(n_epi_warps) * epi_buf_bytes(a.epi);
  // a pair's gate/up epilogue receives the partner's half of the tokens here
  const uint32_t x_bytes = (pair && a.epi == 0) ? 128u * p.xs * 4u : 0u;
  const uint32_t fixed =
      1024u /*align slack*/ + meta_bytes + 512u /*barriers*/ + 128u /*static*/ + epi_bytes + x_bytes;
  const uint32_t a_stage = p.a_slot;  // weight blocks of one K chunk
  const char* env_stages = std::getenv("MXMOE_STAGES");  // tuning override (only lowers)
  auto plan = [&](int kps, int* acc_bufs, uint32_t* sf_col0) {
    // two accumulator buffers (the epilogue of one tile overlaps the next
    // tile's MMAs) whenever they leave tensor memory for two stages of scales
    *acc_bufs = (2u * p.acc_cols + 2u * p.sfc * kps <= kTmemCols) ? 2 : 1;
    *sf_col0 = static_cast<uint32_t>(*acc_bufs) * p.acc_cols;
    if (*sf_col0 + 2u * p.sfc * kps > kTmemCols) return 0;
    const uint32_t per_stage = (a_stage + static_cast<uint32_t>(p.brows) * p.b_row) * static_cast<uint32_t>(kps);
    if (static_cast<uint32_t>(max_smem) <= fixed) return 0;
    int st = static_cast<int>((static_cast<uint32_t>(max_smem) - fixed) / per_stage);
    if (st > kMaxStages) st = kMaxStages;
    if (env_stages) {
      const int v = std::atoi(env_stages);
      if (v >= 2 && v < st) st = v;
    }
    const int tmem_room = static_cast<int>((kTmemCols - *sf_col0) / (p.sfc * kps));
    if (st > tmem_room) st = tmem_room;
    return st >= 2 ? st : 0;
  };
  // Two 128-wide K chunks per pipeline stage when two such stages fit: the
  // fixed per-stage costs of the single MMA-issuing thread (barrier wait,
  // fence, commit) are then paid once per 256 K.
  p.kps = 1;
  if ((p.K / 128) % 2 == 0) {
    int ab;
    uint32_t sc;
    if (plan(2, &ab, &sc) >= 2) p.kps = 2;
  }
  // one row block a tile: single-chunk stages (five in flight at 192 rows
  // measured ahead of two double-chunk stages)
  if (p.one) p.kps = 1;
  if (const char* env = std::getenv(a.epi == 1 && std::getenv("MXMOE_KPS2") ? "MXMOE_KPS2" : "MXMOE_KPS")) {
    const int v = std::atoi(env);
    // four chunks a stage only with packed E2M1 operands (whose MMA loop takes any count)
    if (v == 1 || ((v == 2 || (v == 4 && p.a4)) && (p.K / 128) % v == 0)) p.kps = v;
  }
  const int stages = plan(p.kps, &p.acc_bufs, &p.sf_col0);
  if (stages < 2) return cudaErrorInvalidConfiguration;
  p.stages = stages;
  uint32_t off = 0;
  p.off_a = off;
  off += static_cast<uint32_t>(stages * p.kps) * a_stage;
  p.off_b = off;
  off += static_cast<uint32_t>(stages * p.kps) * p.brows * p.b_row;
  p.off_meta = off;
  off += meta_bytes;
  p.off_bar = off;
  off += 512u;
  p.off_epi = off;
  off += epi_bytes;
  p.off_x = off;
  off += x_bytes;
  const size_t smem = static_cast<size_t>(off) + 1024u;

  // tensor maps
  CUtensorMap tm_a, tm_b;
  {
    // prepared blocks as [expert * NK + K chunk][row block][128 rows][128 K]:
    // one box is a stage's row blocks (the tile's two, one per CTA of a pair)
    // of kps consecutive K chunks
    const size_t nchunk = static_cast<size_t>(a.E + 1) * p.NK;
    // packed E2M1 for kind::mxf4: each block 128 rows of 64 bytes, as bytes
    const cuuint64_t inner = a.a4 ? 64 : 128;
    cuuint64_t dims[4] = {inner, 128, static_cast<cuuint64_t>(p.RB), static_cast<cuuint64_t>(nchunk)};
    cuuint64_t strides[3];
    cuuint32_t box[4] = {static_cast<cuuint32_t>(inner), 128, (pair || p.one) ? 1u : 2u, static_cast<cuuint32_t>(p.kps)};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUtensorMapDataType dt;
    const cuuint64_t blk_bytes = a.fmt == MX_E4M3 ? 16384 : 8192;
    if (a.fmt == MX_E4M3 || a.a4) {
      dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
      strides[0] = inner;
    } else {
      dt = CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
      strides[0] = 64;
    }
    strides[1] = blk_bytes;
    strides[2] = blk_bytes * static_cast<cuuint64_t>(p.RB);
    CUresult r = encode(&tm_a, dt, 4, const_cast<void*>(a.w_prep), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, a.a4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    // gather4: the activation matrix [T, H], four token rows at a time (box one
    // row high); otherwise slot-ordered rows [n_rows, K], one box of `brows`
    // rows per stage (bn, or half of it for each CTA of a pair)
    // (packed E2M1 rows: K/2 bytes, 64 per K chunk)
    const cuuint64_t b_rows = static_cast<cuuint64_t>(p.gather4 ? a.T : a.n_rows);
    const cuuint64_t row_bytes = a.a4 ? static_cast<cuuint64_t>(p.K / 2) : static_cast<cuuint64_t>(p.K);
    cuuint64_t dims[2] = {row_bytes, b_rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {a.a4 ? 64u : 128u, p.gather4 ? 1u : static_cast<cuuint32_t>(p.brows)};
    cuuint32_t es[2] = {1, 1};
    CUresult r = encode(&tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.b_codes), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        a.a4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }

  const bool bt = a.b_scales_t != nullptr;
  const bool narrow = a.bn <= 64 && !pair && !bt;
  void (*kernel)(GemmParams, CUtensorMap, CUtensorMap) =
      narrow ? (a.a4 ? k_grouped_gemm<false, false, -1, 1> : k_grouped_gemm<false, false, -1, 0>)
      : a.epi == 0 ? (pair ? (bt ? k_grouped_gemm<true, true, 0> : k_grouped_gemm<true, false, 0>)
                           : (bt ? k_grouped_gemm<false, true, 0> : k_grouped_gemm<false, false, 0>))
                   : (pair ? k_grouped_gemm<true, false, 1> : k_grouped_gemm<false, false, 1>);
  // the shared-memory opt-in is per device and kernel and only ever raised:
  // skip the driver call when a launch on this device already allowed this much
  {
    static std::atomic<int> smem_allowed[8][kMaxDevices];
    const int which = narrow ? 6 + (a.a4 ? 1 : 0) : a.epi == 0 ? (pair ? 2 : 0) + (bt ? 1 : 0) : 4 + (pair ? 1 : 0);
    std::atomic<int>* allowed = (dev >= 0 && dev < kMaxDevices) ? &smem_allowed[which][dev] : nullptr;
    if (!allowed || allowed->load(std::memory_order_relaxed) < static_cast<int>(smem)) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      if (allowed) allowed->store(static_cast<int>(smem), std::memory_order_relaxed);
    }
  }
  // upper bound on work units: NM * sum_e ceil(count_e / bn) <= NM * (E + 1 + rows / bn)
  const long long bound =
      static_cast<long long>(p.NM) * (p.n_exp + (a.n_rows + p.bn - 1) / p.bn);
  int units = sm_count_gemm() / (pair ? 2 : 1);
  if (bound < units) units = static_cast<int>(bound > 0 ? bound : 1);
  const int grid = units * (pair ? 2 : 1);
  const int timed = timer_begin(a.epi, stream);
  if (!a.pdl && !pair) {
    kernel<<<grid, gemm_threads(pair, bt, a.epi), smem, stream>>>(p, tm_a, tm_b);
    const cudaError_t e = cudaGetLastError();
    timer_end(timed, stream);
    return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(gemm_threads(pair, bt, a.epi));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (a.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (pair) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p, tm_a, tm_b);
  timer_end(timed, stream);
  return e;
}

}  // namespace mxk
