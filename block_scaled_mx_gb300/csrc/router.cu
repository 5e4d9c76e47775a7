// Router GEMM with top-k in its epilogue, on tcgen05 tensor cores (sm_103a):
//
//   logits[t, e] = sum_h x[t, h] * Wr[e, h]     (bf16 x bf16, fp32 accumulation)
//   ids[t, :]    = the k experts with the largest logit + bias[e] (fp32 score),
//                  lowest index on ties, in descending score order
//   w[t, :]      = softmax of the chosen experts' unbiased logits
//
// One CTA per 128-token tile.  Tokens are the MMA's M = 128 rows and experts
// its N columns (up to 256 per instruction, E <= 512 in all), so after the K
// loop each TMEM lane holds one token's whole logit row: every epilogue thread
// selects its own token's top-k in registers, with no cross-thread traffic.
//
// Warp roles (192 threads): warp 0 TMA producer (x tile and router-weight
// tile per 64-wide K chunk, 128-byte swizzle), warp 1 TMEM allocation and the
// single MMA-issuing thread (kind::f16, bf16 operands), warps 2-5 epilogue
// (TMEM lane quarters 2, 3, 0, 1).  Every wait is bounded by wall time; a wait
// that runs out sets MX_ERR_TIMEOUT in the status word and the roles unwind.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "select.cuh"

namespace mxk {

namespace {

constexpr int kRThreads = 192;
constexpr int kRKmax = 16;        // largest k the epilogue selects
constexpr int kRMaxStages = 6;
constexpr int kRMaxDevices = 64;

struct RouterParams {
  int T, H, E, k;
  int n_pad;             // the MMA's N: E rounded up to 16 (512 past 256); padding columns are zero
  int nk;                // 64-wide K chunks
  int stages;
  const float* bias;     // [E] or null
  float* logits;         // [T, E] or null
  int32_t* ids;          // [T, k] or null (logits only)
  float* topk_w;         // [T, k]
  int* status;
  unsigned long long wait_limit_ns;
  uint32_t off_b, off_bar;
  uint32_t a_bytes, b_bytes;  // one stage's x tile and weight tile
  uint32_t tmem_cols;
};

// D[tmem] (+)= A x B for bf16 A (M x 16) and B (16 x N), fp32 accumulation.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t desc_hi,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 ad, bd;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "mov.b64 ad, {%1, %5};\n\t"
      "mov.b64 bd, {%2, %5};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(desc_hi));
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, both
// operands K-major: D format in bits 4-5 (1 = f32), A and B formats in bits
// 7-9 and 10-12 (1 = bf16), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ __forceinline__ uint32_t idesc_bf16(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (((N >> 3) & 0x3Fu) << 17) | (((M >> 4) & 0x1Fu) << 24);
}

// Bounded wait that polls without a suspend hint: the producer and the MMA
// thread resume the moment a stage lands or frees (a suspended thread can
// sleep well past the arrival that completes the phase).
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, unsigned long long limit, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit) {
      set_status(status, MX_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(kRThreads, 1)
    k_router(const __grid_constant__ RouterParams p, const __grid_constant__ CUtensorMap tm_x,
             const __grid_constant__ CUtensorMap tm_w) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + p.off_bar);
  uint64_t* empty = full + S;
  uint64_t* acc = full + 2 * S;
  uint64_t* drain = full + 2 * S + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 2 * S + 2);
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc), 1);
    mbar_init(smem_u32(drain), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int row0 = blockIdx.x * 128;
  const int nk = p.nk;
  const unsigned long long lim = p.wait_limit_ns;

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_x);
      prefetch_tensormap(&tm_w);
      int issued = 0;
      for (int kc = 0; kc < nk; ++kc) {
        const int s = kc % S;
        if (!bounded_wait(smem_u32(&empty[s]), ((kc / S) & 1) ^ 1u, lim, p.status)) break;
        const uint32_t bar = smem_u32(&full[s]);
        mbar_arrive_expect_tx(bar, p.a_bytes + p.b_bytes);
        tma_load_2d(smem_u32(base + s * p.a_bytes), &tm_x, kc * 64, row0, bar);
        uint8_t* b_s = base + p.off_b + s * p.b_bytes;
        for (int n0 = 0; n0 < p.n_pad; n0 += 256) tma_load_2d(smem_u32(b_s + n0 * 128), &tm_w, kc * 64, n0, bar);
        ++issued;
      }
      // every fill issued has landed before the CTA exits
      for (int i = issued > S ? issued - S : 0; i < issued; ++i)
        mbar_wait(smem_u32(&full[i % S]), (i / S) & 1u, 100000000ull);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint32_t a_lo0 = desc_lo_sw128(smem_u32(base));
      const uint32_t b_lo0 = desc_lo_sw128(smem_u32(base + p.off_b));
      uint32_t accum = 0;
      bool ok = true;
      for (int kc = 0; kc < nk && ok; ++kc) {
        const int s = kc % S;
        if (!bounded_wait(smem_u32(&full[s]), (kc / S) & 1u, lim, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_lo = a_lo0 + static_cast<uint32_t>(s) * (p.a_bytes >> 4);
        const uint32_t b_lo = b_lo0 + static_cast<uint32_t>(s) * (p.b_bytes >> 4);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {  // four K = 16 steps of 32 bytes inside the 128-byte row
          for (int n0 = 0; n0 < p.n_pad; n0 += 256) {
            const uint32_t nsz = static_cast<uint32_t>(min(256, p.n_pad - n0));
            mma_bf16(tbase + static_cast<uint32_t>(n0), a_lo + 2u * ks, b_lo + static_cast<uint32_t>(n0) * (128u >> 4) + 2u * ks,
                     kDescHiSw128, idesc_bf16(128, nsz), accum);
          }
          accum = 1u;
        }
        mma_commit(smem_u32(&empty[s]));
      }
      if (ok) mma_commit(smem_u32(acc));
      // every MMA issued has completed before tensor memory is released
      mma_commit(smem_u32(drain));
      mbar_wait(smem_u32(drain), 0, 100000000ull);
    }
  } else {
    // ================================================================ epilogue
    const int q = warp & 3;
    const int t = row0 + 32 * q + lane;
    const bool valid = t < p.T;
    const int E = p.E, k = p.k;
    bool ok = bounded_wait(smem_u32(acc), 0, lim, p.status);
    ok = __all_sync(0xffffffffu, ok) != 0;
    tc_fence_after();
    float sc[kRKmax], lg[kRKmax];
    int id[kRKmax];
#pragma unroll
    for (int j = 0; j < kRKmax; ++j) {
      sc[j] = -INFINITY;
      lg[j] = 0.0f;
      id[j] = -1;
    }
    float thr = -INFINITY;  // the k-th best score so far
    const uint32_t lane_base = tbase + (static_cast<uint32_t>(32 * q) << 16);
    // each thread's 16 logits of a column chunk go through its own 64 bytes of
    // shared memory (the pipeline stages are idle by now), so the selection
    // below runs as one rolled loop: one copy of its code, fetched once
    float* const mine = reinterpret_cast<float*>(base) + (static_cast<size_t>(tid) - 64) * 16;
    for (int c0 = 0; ok && c0 < p.n_pad; c0 += 16) {
      uint32_t v[16];
      __syncwarp();
      tmem_ld_32x32b_x16(lane_base + static_cast<uint32_t>(c0), v);
      tmem_ld_wait();
      if (p.logits && valid) {
        float* row = p.logits + static_cast<size_t>(t) * E;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c0 + i < E) row[c0 + i] = __uint_as_float(v[i]);
      }
      if (!p.ids) continue;
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(mine + i) = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                           __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
#pragma unroll 1
      for (int i = 0; i < 16; ++i) {
        const int e = c0 + i;
        if (e >= E) break;
        const float logit = mine[i];
        const float score = logit + (p.bias ? __ldg(&p.bias[e]) : 0.0f);
        if (score > thr) {
          // insertion into the descending list: the candidate goes in front
          // of the first strictly smaller score (so an equal score stays
          // behind the lower index seen first), and every entry after it
          // shifts down one place
          float cs = score, cl = logit;
          int ci = e;
          bool shifting = false;
#pragma unroll
          for (int j = 0; j < kRKmax; ++j) {
            if (j < k && (shifting || cs > sc[j])) {
              shifting = true;
              const float ts = sc[j], tl = lg[j];
              const int ti = id[j];
              sc[j] = cs;
              lg[j] = cl;
              id[j] = ci;
              cs = ts;
              cl = tl;
              ci = ti;
            }
            if (j == k - 1) thr = sc[j];
          }
        }
      }
    }
    if (ok && p.ids && valid) {
      float vmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < kRKmax; ++j)
        if (j < k) vmax = fmaxf(vmax, lg[j]);
      float ex[kRKmax], sum = 0.0f;
#pragma unroll
      for (int j = 0; j < kRKmax; ++j) {
        ex[j] = j < k ? expf(lg[j] - vmax) : 0.0f;
        sum += ex[j];
      }
#pragma unroll
      for (int j = 0; j < kRKmax; ++j) {
        if (j < k) {
          p.ids[static_cast<size_t>(t) * k + j] = id[j];
          p.topk_w[static_cast<size_t>(t) * k + j] = ex[j] / sum;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tbase, p.tmem_cols);
  }
}

// ------------------------------------------------------------------ small batches
// For a few tokens the router is a matrix-vector product bound by streaming
// the router weights: a block per 2 experts walks H in 256-element chunks,
// four warps per expert, each taking a quarter of every chunk.  The block
// stages each chunk of x (32 tokens x 512 bytes, rows padded by 16 bytes so
// that a quarter-warp's 16-byte loads of 8 rows hit 32 distinct banks; up to
// four such token tiles) and of its experts' rows in shared memory with
// cp.async, three chunks in flight.  Lane t accumulates the dot products of
// tokens t, t + 32, ... over its quarters in fp32 (8 exact products per
// 16-byte step, two interleaved partial sums, the expert's weights a
// broadcast shared-memory read); the four quarters' sums are added in a fixed
// order.  The block that finishes last (a counter it resets; nobody
// waits) selects every token's top-k from the logits in global memory, one
// warp per token.
constexpr int kRSmallMaxT = 128;
constexpr int kRSmallExpertsPerBlock = 2;
constexpr int kRSmallWarpsPerExpert = 4;
constexpr int kRSmallRowWords = 132;  // 512 bytes of x + 16 bytes of padding, in 32-bit words

struct RouterSmallParams {
  const uint4* x;        // bf16 [T, H] as 16-byte groups
  const uint4* w;        // bf16 [E, H]
  const float* bias;
  int T, H, E, k;
  float* logits;         // [T, E] (the caller's, or the workspace's)
  int32_t* ids;          // [T, k] or null
  float* topk_w;
  unsigned* done;        // blocks finished (zero between calls: the last block resets it)
};

// 8 products of bf16 pairs (exact in fp32) added to acc in element order.
__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b, float acc) {
  const uint32_t x[4] = {a.x, a.y, a.z, a.w};
  const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fmaf(__uint_as_float(x[i] << 16), __uint_as_float(w[i] << 16), acc);
    acc = fmaf(__uint_as_float(x[i] & 0xFFFF0000u), __uint_as_float(w[i] & 0xFFFF0000u), acc);
  }
  return acc;
}

// One token's top-k by score = logit + bias (fp32 addition), lowest index on
// equal scores, descending; weights: softmax of the chosen unbiased logits.
// Lane l holds experts l, l + 32, ... as order-preserving score keys; each
// round's winner is two warp reductions (the largest key, then the lowest
// index holding it), its logit taken from the lane that holds it.
template <int PER>
__device__ __forceinline__ void router_select(const RouterSmallParams& p, int t, int lane) {
  const int E = p.E, k = p.k;
  const float* row = p.logits + static_cast<size_t>(t) * E;
  float lg[PER];
  uint32_t key[PER];  // 0: past E
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < E ? __ldcg(&row[e]) : 0.0f;
    key[i] = e < E ? order_key(lg[i] + (p.bias ? __ldg(&p.bias[e]) : 0.0f)) : 0u;
  }
  uint32_t taken = 0;
  float my_l = 0.0f;
  int my_i = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    float bl = 0.0f;
    int bs = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (!((taken >> i) & 1u) && key[i] > bk) {
        bk = key[i];
        bl = lg[i];
        bs = i;
      }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const int bi = static_cast<int>(__reduce_min_sync(0xffffffffu, bk == m && m != 0u
                                                                        ? static_cast<uint32_t>(lane + 32 * bs)
                                                                        : 0xFFFFFFFFu));
    const float wl = __shfl_sync(0xffffffffu, bl, bi & 31);
    if (bi >= 0 && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_l = wl;
      my_i = bi;
    }
  }
  float vmax = lane < k ? my_l : -INFINITY;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
  const float ex = lane < k ? expf(my_l - vmax) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    p.ids[static_cast<size_t>(t) * k + lane] = my_i;
    p.topk_w[static_cast<size_t>(t) * k + lane] = ex / sum;
  }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kRSmallStages = 3;                                   // chunks in flight
constexpr int kRSmallXU4 = 32 * kRSmallRowWords / 4;               // one token tile's x rows, 16-byte units
constexpr int kRSmallTiles = kRSmallMaxT / 32;                     // token tiles one sweep of H carries
// one stage: nt token tiles of x rows, then the block's experts' chunks
__host__ __device__ constexpr int rsmall_stage_u4(int nt) { return nt * kRSmallXU4 + kRSmallExpertsPerBlock * 32; }
__host__ __device__ constexpr size_t rsmall_smem(int nt) {
  return static_cast<size_t>(kRSmallStages) * rsmall_stage_u4(nt) * 16;
}

template <int PER>
__global__ void __launch_bounds__(256) k_router_small(const RouterSmallParams p) {
  extern __shared__ uint4 rsm[];  // kRSmallStages stages
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ew = warp / kRSmallWarpsPerExpert, wq = warp % kRSmallWarpsPerExpert;  // expert of the block, quarter
  const int e = blockIdx.x * kRSmallExpertsPerBlock + ew;
  __shared__ float part[8][32];
  const int T = p.T, H8 = p.H / 8, nch = (H8 + 31) / 32;  // 16-byte groups per row, 256-element chunks
  const int nt = (T + 31) / 32;                          // token tiles (all in one sweep of H)
  const int stage_u4 = rsmall_stage_u4(nt);
  // chunk c into stage c % S: thread i copies groups i, i + 256, ... of each
  // [32 rows][32 groups] x tile, and threads i < 64 group i % 32 of the
  // block's expert i / 32 (zero-filled past T or H); one commit group per
  // chunk, empty ones past the last so that the wait count stays fixed
  auto issue = [&](int c) {
    if (c < nch) {
      uint4* const sd = rsm + (c % kRSmallStages) * stage_u4;
      for (int tt = 0; tt < nt; ++tt) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int i = tid + 256 * r, row = i >> 5, g = c * 32 + (i & 31), t = 32 * tt + row;
          const bool ok = t < T && g < H8;
          cp_async16(smem_u32(sd + tt * kRSmallXU4 + row * (kRSmallRowWords / 4) + (i & 31)),
                     ok ? static_cast<const void*>(&p.x[static_cast<size_t>(t) * H8 + g]) : p.x, ok);
        }
      }
      if (tid < kRSmallExpertsPerBlock * 32) {
        const int ee = min(blockIdx.x * kRSmallExpertsPerBlock + (tid >> 5), p.E - 1);
        const uint4* const wr = p.w + static_cast<size_t>(ee) * H8;
        const bool okw = c * 32 + lane < H8;
        cp_async16(smem_u32(sd + nt * kRSmallXU4 + tid), okw ? &wr[c * 32 + lane] : wr, okw);
      }
    }
    cp_async_commit();
  };
  float acc0[kRSmallTiles], acc1[kRSmallTiles];
#pragma unroll
  for (int tt = 0; tt < kRSmallTiles; ++tt) acc0[tt] = acc1[tt] = 0.0f;
#pragma unroll
  for (int c = 0; c < kRSmallStages - 1; ++c) issue(c);
  const int j0 = wq * (32 / kRSmallWarpsPerExpert);
  for (int c = 0; c < nch; ++c) {
    issue(c + kRSmallStages - 1);
    cp_async_wait<kRSmallStages - 1>();
    __syncthreads();
    const uint4* const st = rsm + (c % kRSmallStages) * stage_u4;
    const uint4* const wr = st + nt * kRSmallXU4 + ew * 32 + j0;
#pragma unroll
    for (int tt = 0; tt < kRSmallTiles; ++tt) {
      if (tt < nt) {
        const uint4* xr = st + tt * kRSmallXU4 + lane * (kRSmallRowWords / 4) + j0;
#pragma unroll
        for (int j = 0; j < 32 / kRSmallWarpsPerExpert; j += 2) {  // groups past H are zero in both
          acc0[tt] = dot8_bf16(xr[j], wr[j], acc0[tt]);
          acc1[tt] = dot8_bf16(xr[j + 1], wr[j + 1], acc1[tt]);
        }
      }
    }
    __syncthreads();  // the stage is refilled by the next iteration's copies
  }
  cp_async_wait<0>();
#pragma unroll
  for (int tt = 0; tt < kRSmallTiles; ++tt) {
    if (tt < nt) {
      part[warp][lane] = acc0[tt] + acc1[tt];
      __syncthreads();
      const int t = 32 * tt + lane;
      if (wq == 0 && e < p.E && t < T) {
        float v = part[warp][lane];
#pragma unroll
        for (int qq = 1; qq < kRSmallWarpsPerExpert; ++qq) v += part[warp + qq][lane];
        p.logits[static_cast<size_t>(t) * p.E + e] = v;
      }
      __syncthreads();
    }
  }
  if (!p.ids) return;
  // the last block to finish selects (its reads of the other blocks' logits
  // follow their fences and the counter)
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) *p.done = 0u;  // ready for the next call
  for (int t = warp; t < T; t += blockDim.x >> 5) router_select<PER>(p, t, lane);
}

PFN_cuTensorMapEncodeTiled_v12000 router_encode_fn() {
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

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  // a few tokens with somewhere to keep the logits: the small-batch kernel
  float* small_logits = a.logits ? a.logits : a.scratch_logits;
  if (a.T <= kRSmallMaxT && small_logits && a.H % 8 == 0) {
    RouterSmallParams q{};
    q.x = static_cast<const uint4*>(a.x);
    q.w = static_cast<const uint4*>(a.w);
    q.bias = a.bias;
    q.T = a.T;
    q.H = a.H;
    q.E = a.E;
    q.k = a.k;
    q.logits = small_logits;
    q.ids = a.ids;
    q.topk_w = a.topk_w;
    q.done = a.counter;
    const unsigned grid = static_cast<unsigned>((a.E + kRSmallExpertsPerBlock - 1) / kRSmallExpertsPerBlock);
    void (*kern)(RouterSmallParams) = a.E <= 32 ? k_router_small<1> : a.E <= 128 ? k_router_small<4> : k_router_small<16>;
    // the shared-memory opt-in, once per device and kernel
    {
      static std::atomic<unsigned> allowed[kRMaxDevices];
      int dev = 0;
      cudaGetDevice(&dev);
      const unsigned bit = a.E <= 32 ? 1u : a.E <= 128 ? 2u : 4u;
      if (dev < 0 || dev >= kRMaxDevices || !(allowed[dev].load(std::memory_order_relaxed) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(rsmall_smem(kRSmallTiles)));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kRMaxDevices) allowed[dev].fetch_or(bit, std::memory_order_relaxed);
      }
    }
    kern<<<grid, 256, rsmall_smem((a.T + 31) / 32), stream>>>(q);
    return cudaGetLastError();
  }
  auto encode = router_encode_fn();
  if (!encode) return cudaErrorNotSupported;
  RouterParams p{};
  p.T = a.T;
  p.H = a.H;
  p.E = a.E;
  p.k = a.k;
  // the MMA's N: E rounded up to 16, or 512 past 256 experts (two full
  // 256-row weight boxes per stage, so each box's byte count is fixed)
  p.n_pad = a.E <= 256 ? (a.E + 15) & ~15 : 512;
  p.nk = a.H / 64;
  p.bias = a.bias;
  p.logits = a.logits;
  p.ids = a.ids;
  p.topk_w = a.topk_w;
  p.status = a.status;
  p.wait_limit_ns = a.wait_limit_ns;
  p.a_bytes = 128u * 128u;                                  // 128 tokens x 64 bf16
  p.b_bytes = static_cast<uint32_t>(p.n_pad) * 128u;        // n_pad experts x 64 bf16
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(p.n_pad)) cols <<= 1;
  p.tmem_cols = cols;
  int dev = 0;
  cudaGetDevice(&dev);
  int max_smem = 0;
  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const uint32_t fixed = 1024u + 256u;
  int stages = static_cast<int>((static_cast<uint32_t>(max_smem) - fixed) / (p.a_bytes + p.b_bytes));
  if (stages > kRMaxStages) stages = kRMaxStages;
  if (stages > p.nk) stages = p.nk;
  if (stages < 1) return cudaErrorInvalidConfiguration;
  p.stages = stages;
  p.off_b = static_cast<uint32_t>(stages) * p.a_bytes;
  p.off_bar = p.off_b + static_cast<uint32_t>(stages) * p.b_bytes;
  const size_t smem = p.off_bar + 256u + 1024u;

  CUtensorMap tm_x, tm_w;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.H), static_cast<cuuint64_t>(a.T)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.H) * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    if (encode(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.x), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.H), static_cast<cuuint64_t>(a.E)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.H) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(p.n_pad < 256 ? p.n_pad : 256)};
    cuuint32_t es[2] = {1, 1};
    if (encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.w), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    static std::atomic<int> smem_allowed[kRMaxDevices];
    if (dev < 0 || dev >= kRMaxDevices || smem_allowed[dev].load(std::memory_order_relaxed) < static_cast<int>(smem)) {
      cudaError_t e = cudaFuncSetAttribute(k_router, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < kRMaxDevices) smem_allowed[dev].store(static_cast<int>(smem), std::memory_order_relaxed);
    }
  }
  const unsigned grid = static_cast<unsigned>((a.T + 127) / 128);
  k_router<<<grid, kRThreads, smem, stream>>>(p, tm_x, tm_w);
  return cudaGetLastError();
}

}  // namespace mxk
