// Memory-bound kernels of the MX MoE layer: activation / weight MX
// quantisation, router top-k with softmax, the device-side token -> expert
// permutation, the activation row gather and the load-time weight re-layout.
//
// All of these are HBM- or launch-latency-bound: 128-bit coalesced loads,
// grid sizes in multiples of the SM count, no tensor cores.
#include <cuda_runtime.h>
#include <cstdint>
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "select.cuh"

namespace mxk {

static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 152;
  }
  return n;
}

static unsigned grid_for(int64_t work_items, int threads, int per_sm) {
  int64_t blocks = (work_items + threads - 1) / threads;
  int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

// ------------------------------------------------------------------ activation quantisation
// One thread = 8 bf16 (one 16-byte load); four consecutive lanes = one MX block
// of 32.  Block amax over the bf16 magnitudes (integer max of the 15-bit
// magnitude is monotonic), shared exponent from its bits, exact scaling by
// 2^-s in fp32, then RNE/saturating E4M3 encoding.
__device__ __forceinline__ void quantize_act_step(const uint4* __restrict__ x, int64_t n8, int64_t i,
                                                  int lane, uint2* __restrict__ codes,
                                                  uint8_t* __restrict__ scales) {
  const bool valid = i < n8;
  const uint4 v = valid ? __ldg(&x[i]) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t amax = 0;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    amax = max(amax, w[m] & 0x7FFFu);
    amax = max(amax, (w[m] >> 16) & 0x7FFFu);
  }
  amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int s = mx_block_exponent(amax << 16, 8);
  const float p = pow2_neg(s);
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t c01 = enc_e4m3x2(__uint_as_float(w[m] << 16) * p, __uint_as_float(w[m] & 0xFFFF0000u) * p);
    packed[m >> 1] |= c01 << ((m & 1) * 16);
  }
  if (valid) {
    codes[i] = make_uint2(packed[0], packed[1]);
    if ((lane & 3) == 0) scales[i >> 2] = static_cast<uint8_t>(s + 127);
  }
}

// The same for MXFP4 activations: shared exponent with emax 2 (E2M1), codes
// packed two per byte, element 2i in the low nibble (one 32-bit word of 8 codes
// per thread).
__device__ __forceinline__ void quantize_act_step_e2m1(const uint4* __restrict__ x, int64_t n8, int64_t i,
                                                       int lane, uint32_t* __restrict__ codes,
                                                       uint8_t* __restrict__ scales) {
  const bool valid = i < n8;
  const uint4 v = valid ? __ldg(&x[i]) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t amax = 0;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    amax = max(amax, w[m] & 0x7FFFu);
    amax = max(amax, (w[m] >> 16) & 0x7FFFu);
  }
  amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int s = mx_block_exponent(amax << 16, 2);
  const float p = pow2_neg(s);
  uint32_t packed = 0u;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    packed |= enc_e2m1(__uint_as_float(w[m] << 16) * p) << (8 * m);
    packed |= enc_e2m1(__uint_as_float(w[m] & 0xFFFF0000u) * p) << (8 * m + 4);
  }
  if (valid) {
    codes[i] = packed;
    if ((lane & 3) == 0) scales[i >> 2] = static_cast<uint8_t>(s + 127);
  }
}

template <bool E2M1>
__global__ void __launch_bounds__(256) k_quantize_act(const uint4* __restrict__ x, int64_t n8, void* __restrict__ codes,
                                                      uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i - lane < n8;
       i += stride) {
    if (E2M1) quantize_act_step_e2m1(x, n8, i, lane, static_cast<uint32_t*>(codes), scales);
    else quantize_act_step(x, n8, i, lane, static_cast<uint2*>(codes), scales);
  }
}

cudaError_t launch_quantize_act(const void* x, int64_t n_elems, uint8_t* codes, uint8_t* scales,
                                cudaStream_t s, int fmt) {
  const int64_t n8 = n_elems / 8;
  if (n8 == 0) return cudaSuccess;
  if (fmt == MX_E2M1)
    k_quantize_act<true><<<grid_for(n8, 256, 8), 256, 0, s>>>(static_cast<const uint4*>(x), n8, codes, scales);
  else
    k_quantize_act<false><<<grid_for(n8, 256, 8), 256, 0, s>>>(static_cast<const uint4*>(x), n8, codes, scales);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ weight quantisation
// One thread = 4 fp32 (one 16-byte load); eight consecutive lanes = one block.
__global__ void __launch_bounds__(256) k_quantize_weights(const float4* __restrict__ w, int64_t n4,
                                                          int fmt, uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int emax = fmt == MX_E4M3 ? 8 : 2;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i - lane < n4;
       i += stride) {
    const bool valid = i < n4;
    const float4 v = valid ? __ldg(&w[i]) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float f[4] = {v.x, v.y, v.z, v.w};
    uint32_t amax = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) amax = max(amax, __float_as_uint(f[m]) & 0x7FFFFFFFu);
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const int s = mx_block_exponent(amax, emax);
    const float p = pow2_neg(s);
    if (valid) {
      if (fmt == MX_E4M3) {
        uint32_t packed = 0;
#pragma unroll
        for (int m = 0; m < 4; m += 2) packed |= enc_e4m3x2(f[m] * p, f[m + 1] * p) << (8 * m);
        reinterpret_cast<uint32_t*>(codes)[i] = packed;
      } else {
        uint32_t packed = 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) packed |= enc_e2m1(f[m] * p) << (4 * m);
        reinterpret_cast<uint16_t*>(codes)[i] = static_cast<uint16_t>(packed);
      }
      if ((lane & 7) == 0) scales[i >> 3] = static_cast<uint8_t>(s + 127);
    }
  }
}

cudaError_t launch_quantize_weights(const float* w, int64_t n_elems, int fmt, uint8_t* codes,
                                    uint8_t* scales, cudaStream_t s) {
  const int64_t n4 = n_elems / 4;
  if (n4 == 0) return cudaSuccess;
  k_quantize_weights<<<grid_for(n4, 256, 8), 256, 0, s>>>(reinterpret_cast<const float4*>(w), n4,
                                                          fmt, codes, scales);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ router top-k
// One warp per token.  Lane l holds logits l, l+32, ... in registers as
// order-preserving 32-bit keys (sign-magnitude floats mapped onto unsigned
// order; -0 folded into +0 first, so equal logits give equal keys).  Each of
// the k rounds takes the warp-wide maximum key among the logits not yet taken
// (one warp reduction), then the lowest expert index holding it (a second):
// larger logit, then lower index.  Lane j keeps round j's winner, so ids come
// out in descending-logit order; softmax over the k winners in fp32.
template <int PER>
__device__ __forceinline__ void topk_token(const float* __restrict__ logits, int t, int E, int k,
                                           int lane, int32_t* __restrict__ ids,
                                           float* __restrict__ wout) {
  const float* row = logits + static_cast<int64_t>(t) * E;
  uint32_t key[PER];  // 0: past E (below every logit's key, -inf's included)
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? order_key(__ldg(&row[e])) : 0u;
  }
  uint32_t taken = 0;
  uint32_t my_key = 0;
  int my_i = 0;
  for (int j = 0; j < k; ++j) {
    // this lane's best untaken key; on equal keys the lower i (lower index)
    uint32_t bk = 0;
    int bl = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (!((taken >> i) & 1u) && key[i] > bk) {
        bk = key[i];
        bl = i;
      }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const int bi = static_cast<int>(__reduce_min_sync(0xffffffffu, bk == m && m != 0u
                                                                        ? static_cast<uint32_t>(lane + 32 * bl)
                                                                        : 0xFFFFFFFFu));
    if (bi >= 0 && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_key = m;
      my_i = bi;
    }
  }
  const float my_v = key_value(my_key);
  const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
  float ex = lane < k ? expf(my_v - vmax) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    ids[static_cast<int64_t>(t) * k + lane] = my_i;
    wout[static_cast<int64_t>(t) * k + lane] = ex / sum;
  }
}

template <int PER>
__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int T, int E, int k,
                                              int32_t* __restrict__ ids, float* __restrict__ wout) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  topk_token<PER>(logits, t, E, k, threadIdx.x & 31, ids, wout);
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((T + 7) / 8);
  if (E <= 32) k_topk<1><<<blocks, 256, 0, s>>>(logits, T, E, k, ids, w);
  else if (E <= 128) k_topk<4><<<blocks, 256, 0, s>>>(logits, T, E, k, ids, w);
  else if (E <= 512) k_topk<16><<<blocks, 256, 0, s>>>(logits, T, E, k, ids, w);
  else k_topk<32><<<blocks, 256, 0, s>>>(logits, T, E, k, ids, w);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ permutation
// Stable counting sort of the T*k routed slots by expert, with the T shared
// slots appended, without atomics whose order could leak into the result:
//  pass 1 (one block per chunk of 256 tokens): per warp, a bitmask per expert
//    of the lanes (tokens) routed to it; a slot's rank inside its chunk is the
//    popcount of lower lanes plus the popcounts of earlier warps.  The block
//    writes its per-expert counts; the last block to finish (threadfence +
//    counter) sums them into counts / offsets and turns them into per-chunk
//    bases (experts ascending, chunks ascending).
//  pass 2: each slot lands at chunk_base + rank.
// With a single chunk, pass 1 finishes the scatter itself.
size_t permute_scratch_bytes(int T, int E, int k) {
  const size_t nchunks = static_cast<size_t>((T + kPermuteChunk - 1) / kPermuteChunk);
  auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  return al(256) + al(nchunks * E * 4) * 2 + al(static_cast<size_t>(T) * k * 4) + al(256);
}

PermuteScratch permute_scratch_carve(void* ws, int T, int E, int k) {
  const size_t nchunks = static_cast<size_t>((T + kPermuteChunk - 1) / kPermuteChunk);
  auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  uint8_t* p = static_cast<uint8_t*>(ws);
  PermuteScratch sc;
  sc.status = reinterpret_cast<int*>(p);
  p += al(256);
  sc.chunk_counts = reinterpret_cast<int*>(p);
  p += al(nchunks * E * 4);
  sc.chunk_base = reinterpret_cast<int*>(p);
  p += al(nchunks * E * 4);
  sc.local_rank = reinterpret_cast<int*>(p);
  p += al(static_cast<size_t>(T) * k * 4);
  sc.done = reinterpret_cast<unsigned*>(p);
  return sc;
}

// Dynamic shared memory of one permutation block: per warp and expert the
// lane masks and their exclusive prefix over warps, E + 2 ints of scan space,
// and the ids of the block's tokens.
static size_t permute_block_smem(int T, int E, int k) {
  const int nt = T < kPermuteChunk ? T : kPermuteChunk;
  return (static_cast<size_t>(2 * (kPermuteChunk / 32)) * E + (E + 2) + static_cast<size_t>(nt) * k) * 4;
}

// One chunk of pass 1 (and, for a single chunk, the whole permutation), run by
// one block of kPermuteChunk threads.  The loops over a token's k slots stay
// rolled and read the ids from shared memory: this code runs once per call, in
// one block, right after other kernels have streamed far more than L2 holds,
// so its instructions come from DRAM and its length, not its arithmetic, sets
// its latency.
__device__ __forceinline__ void permute_count_block(const int32_t* __restrict__ ids, int T, int E,
                                                    int k, int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ sorted_slot,
                                                    const PermuteScratch& sc, int nchunks, int chunk,
                                                    uint32_t* bits) {
  constexpr int kWarps = kPermuteChunk / 32;
  __shared__ int s_is_last;
  __shared__ int s_warp_tot[kWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* const pre = bits + kWarps * E;                   // [warp][E]: lanes of earlier warps
  int* const scan = reinterpret_cast<int*>(pre + kWarps * E);  // E + 2
  int* const s_ids = scan + E + 2;                            // [token of the chunk][k]
  const int t0 = chunk * kPermuteChunk;
  const int nt = min(kPermuteChunk, T - t0);
  const int n_ids = nt * k;
  // the chunk's ids into shared memory, eight coalesced loads in flight per thread
  const int32_t* const src = ids + static_cast<int64_t>(t0) * k;
  for (int i0 = 0; i0 < n_ids; i0 += 8 * kPermuteChunk) {
    int v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kPermuteChunk + tid;
      v[u] = i < n_ids ? __ldcg(src + i) : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kPermuteChunk + tid;
      if (i < n_ids) s_ids[i] = v[u];
    }
  }
  for (int i = tid; i < kWarps * E; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  const int t = t0 + tid;
  const bool valid = tid < nt;
  int* const my_ids = s_ids + tid * k;
  // per warp and expert, the lanes (tokens) routed to it; an id out of range
  // is reported and its slot dropped
  if (valid) {
    for (int j = 0; j < k; ++j) {
      const int e = my_ids[j];
      if (e < 0 || e >= E) {
        set_status(sc.status, MX_ERR_DEVICE_ARG);
        my_ids[j] = -1;
      } else {
        atomicOr(&bits[warp * E + e], 1u << lane);
      }
    }
  }
  __syncthreads();
  // per expert: the chunk's count and each warp's offset inside it
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < kWarps; ++w) {
      pre[w * E + e] = c;
      c += __popc(bits[w * E + e]);
    }
    scan[e] = c;
    if (nchunks > 1) sc.chunk_counts[static_cast<int64_t>(chunk) * E + e] = c;
  }
  __syncthreads();
  // a slot's rank among the chunk's slots of its expert: earlier warps, then lower lanes
  const uint32_t lt = (1u << lane) - 1u;
  if (nchunks > 1) {
    if (valid)
      for (int j = 0; j < k; ++j) {
        const int e = my_ids[j];
        if (e >= 0)
          sc.local_rank[static_cast<int64_t>(t) * k + j] =
              static_cast<int>(pre[warp * E + e]) + __popc(bits[warp * E + e] & lt);
      }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_is_last = (atomicAdd(sc.done, 1u) == static_cast<unsigned>(nchunks - 1));
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    // the last block: per-expert totals over all chunks (eight loads in flight)
    for (int e = tid; e < E; e += blockDim.x) {
      int c = 0, ch = 0;
      for (; ch + 8 <= nchunks; ch += 8) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldcg(&sc.chunk_counts[static_cast<int64_t>(ch + u) * E + e]);
#pragma unroll
        for (int u = 0; u < 8; ++u) c += v[u];
      }
      for (; ch < nchunks; ++ch) c += __ldcg(&sc.chunk_counts[static_cast<int64_t>(ch) * E + e]);
      scan[e] = c;
    }
  }
  if (tid == 0) scan[E] = T;  // the shared expert: every token once
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) counts[e] = scan[e];
  // block-wide exclusive scan of scan[0..E] (E+1 <= 1025 values): each thread
  // owns a contiguous run, warp shuffles scan the run totals.
  const int n = E + 1;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int b0 = min(tid * per, n), b1 = min(b0 + per, n);
  int run = 0;
  for (int i = b0; i < b1; ++i) run += scan[i];
  int incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) s_warp_tot[warp] = incl;
  __syncthreads();
  int warp_base = 0;
  for (int w = 0; w < warp; ++w) warp_base += s_warp_tot[w];
  int acc = warp_base + incl - run;
  __syncthreads();
  for (int i = b0; i < b1; ++i) {
    const int c = scan[i];
    scan[i] = acc;
    acc += c;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) offsets[e] = scan[e];
  if (tid == 0) offsets[E + 1] = T * (k + 1);
  if (nchunks > 1) {
    for (int e = tid; e < E; e += blockDim.x) {
      int base = scan[e];
      int ch = 0;
      for (; ch + 8 <= nchunks; ch += 8) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldcg(&sc.chunk_counts[static_cast<int64_t>(ch + u) * E + e]);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          sc.chunk_base[static_cast<int64_t>(ch + u) * E + e] = base;
          base += v[u];
        }
      }
      for (; ch < nchunks; ++ch) {
        sc.chunk_base[static_cast<int64_t>(ch) * E + e] = base;
        base += __ldcg(&sc.chunk_counts[static_cast<int64_t>(ch) * E + e]);
      }
    }
  } else if (valid) {
    // single chunk: scatter directly (this block holds every token)
    for (int j = 0; j < k; ++j) {
      const int e = my_ids[j];
      if (e >= 0)
        sorted_slot[scan[e] + static_cast<int>(pre[warp * E + e]) + __popc(bits[warp * E + e] & lt)] =
            t * (k + 1) + j;
    }
    sorted_slot[scan[E] + t] = t * (k + 1) + k;
  }
}

__global__ void __launch_bounds__(kPermuteChunk) k_permute_count(
    const int32_t* __restrict__ ids, int T, int E, int k, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_slot, PermuteScratch sc,
    int nchunks) {
  extern __shared__ uint32_t bits[];
  permute_count_block(ids, T, E, k, counts, offsets, sorted_slot, sc, nchunks, blockIdx.x, bits);
}

__global__ void __launch_bounds__(kPermuteChunk) k_permute_scatter(
    const int32_t* __restrict__ ids, int T, int E, int k, const int32_t* __restrict__ offsets,
    int32_t* __restrict__ sorted_slot, PermuteScratch sc) {
  const int chunk = blockIdx.x;
  const int t = chunk * kPermuteChunk + threadIdx.x;
  if (blockIdx.x == 0 && threadIdx.x == 0) *sc.done = 0u;  // ready for the next call
  if (t >= T) return;
  for (int j = 0; j < k; ++j) {
    const int e = ids[static_cast<int64_t>(t) * k + j];
    if (e < 0 || e >= E) continue;
    const int pos = sc.chunk_base[static_cast<int64_t>(chunk) * E + e] +
                    sc.local_rank[static_cast<int64_t>(t) * k + j];
    sorted_slot[pos] = t * (k + 1) + j;
  }
  sorted_slot[offsets[E] + t] = t * (k + 1) + k;
}

cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* sorted_slot, const PermuteScratch& sc,
                           cudaStream_t s) {
  const int nchunks = T == 0 ? 1 : (T + kPermuteChunk - 1) / kPermuteChunk;
  const size_t smem = permute_block_smem(T, E, k);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_permute_count, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  k_permute_count<<<nchunks, kPermuteChunk, smem, s>>>(ids, T, E, k, counts, offsets, sorted_slot, sc,
                                                       nchunks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || nchunks == 1) return e;
  k_permute_scatter<<<nchunks, kPermuteChunk, 0, s>>>(ids, T, E, k, offsets, sorted_slot, sc);
  e = cudaGetLastError();
  // the counting pass ran and left its last-block counter at nchunks; the
  // scatter, which puts it back to zero, did not start: reset it here so the
  // next call on this workspace still finds its last block
  if (e != cudaSuccess) cudaMemsetAsync(sc.done, 0, sizeof(unsigned), s);
  return e;
}

// ------------------------------------------------------------------ fused prologue
// The first launch of the fused layer: every block routes its share of tokens
// (warp per token), quantises its share of x and zeroes its share of out; with
// `permute` set, the last block to finish (threadfence + counter: nobody waits)
// computes the whole permutation, which needs T <= kPermuteChunk.  It lets the
// next grid (the gate/up GEMM, launched programmatically dependent) start its
// set-up at once.
// E2M1: quantise to MXFP4 (one instantiation per activation format: the
// first launch of a layer runs its code cold).
template <int PER, bool PERMUTE, bool E2M1>
__global__ void __launch_bounds__(kPermuteChunk) k_prologue(PrologueArgs a) {
  extern __shared__ uint32_t bits[];
  __shared__ int s_last;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int t = blockIdx.x * (kPermuteChunk / 32) + warp; t < a.T; t += gridDim.x * (kPermuteChunk / 32))
    topk_token<PER>(a.logits, t, a.E, a.k, lane, a.ids, a.topk_w);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid;
  if (E2M1)
    for (int64_t i = first; i - lane < a.n8; i += stride)
      quantize_act_step_e2m1(a.x, a.n8, i, lane, reinterpret_cast<uint32_t*>(a.codes), a.scales);
  else
    for (int64_t i = first; i - lane < a.n8; i += stride) quantize_act_step(a.x, a.n8, i, lane, a.codes, a.scales);
  for (int64_t i = first; i < a.n_out4; i += stride) a.out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!PERMUTE) return;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.sc.done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  permute_count_block(a.ids, a.T, a.E, a.k, a.counts, a.offsets, a.sorted_slot, a.sc, 1, 0, bits);
  if (tid == 0) *a.sc.done = 0u;  // ready for the next call
}

cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t s) {
  const int64_t work = a.n8 > a.n_out4 ? a.n8 : a.n_out4;
  int64_t blocks = (work + kPermuteChunk - 1) / kPermuteChunk;
  const int64_t route_blocks = (a.T + kPermuteChunk / 32 - 1) / (kPermuteChunk / 32);
  if (blocks < route_blocks) blocks = route_blocks;
  // eight 256-thread blocks per SM keep enough 16-byte loads in flight for
  // the quantisation stream of a large batch
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const size_t smem = a.permute ? permute_block_smem(a.T, a.E, a.k) : 0;
  const unsigned g = static_cast<unsigned>(blocks);
  void (*kern)(PrologueArgs);
  if (a.act_e2m1) {
    if (a.permute)
      kern = a.E <= 32 ? k_prologue<1, true, true> : a.E <= 128 ? k_prologue<4, true, true>
           : a.E <= 512 ? k_prologue<16, true, true> : k_prologue<32, true, true>;
    else
      kern = a.E <= 32 ? k_prologue<1, false, true> : a.E <= 128 ? k_prologue<4, false, true>
           : a.E <= 512 ? k_prologue<16, false, true> : k_prologue<32, false, true>;
  } else {
    if (a.permute)
      kern = a.E <= 32 ? k_prologue<1, true, false> : a.E <= 128 ? k_prologue<4, true, false>
           : a.E <= 512 ? k_prologue<16, true, false> : k_prologue<32, true, false>;
    else
      kern = a.E <= 32 ? k_prologue<1, false, false> : a.E <= 128 ? k_prologue<4, false, false>
           : a.E <= 512 ? k_prologue<16, false, false> : k_prologue<32, false, false>;
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<g, kPermuteChunk, smem, s>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ prologue of a large batch
// The first launch of the layer for T > kPermuteChunk: one grid whose blocks
// are all resident at once (its size comes from the occupancy query) runs, with
// a grid barrier (a global counter, bounded waits) between the phases:
//   0. routing (warp per token);
//   1. the chunked permutation's first pass, one block per chunk of 256
//      tokens, the last of them (counter, nobody waits) turning the per-chunk
//      counts into the expert offsets and chunk bases; the other blocks
//      quantise x meanwhile;
//   2. the scatter of every slot to its position; the other blocks zero out;
//   3. (wide schedule) the copy of each slot's activation row into slot
//      order, the B operand the wide gate/up GEMM loads as 2-D boxes, and of
//      its scales into K-chunk-major order.
// Together with the two grouped GEMMs the layer is then three launches.
namespace {
__device__ bool grid_barrier(unsigned* bar, unsigned target, int* status, unsigned long long limit_ns) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    int ok = 1;
    const uint64_t t0 = globaltimer_ns();
    while (*reinterpret_cast<volatile unsigned*>(bar) < target) {
      if (globaltimer_ns() - t0 > limit_ns) {
        set_status(status, MX_ERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(128);
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}
}  // namespace

// Scale words of slot-ordered rows, K-chunk-major (the grouped GEMM's scale
// warps then read a chunk's words of consecutive rows in one coalesced load):
// dst_sc[c * n_rows + p] = src_sc[t * words + c], t the token of slot position p.
// A work item is one slot and a run of 8 words (consecutive items: consecutive
// slots, so a warp's stores of one word are one 128-byte run); two loads in
// flight per thread keep the register count of the kernels it sits in.
__device__ __forceinline__ void gather_scales_t(const uint32_t* __restrict__ src_sc, int T, int words,
                                                const int32_t* __restrict__ sorted_slot, int k, int n_rows,
                                                uint32_t* __restrict__ dst_sc, int64_t first, int64_t stride) {
  const int64_t items = static_cast<int64_t>(n_rows) * ((words + 7) / 8);
  for (int64_t i = first; i < items; i += stride) {
    const int g = static_cast<int>(i / n_rows);
    const int p = static_cast<int>(i - static_cast<int64_t>(g) * n_rows);
    const int t = __ldcg(&sorted_slot[p]) / (k + 1);
    const bool ok = t >= 0 && t < T;
    const uint32_t* row = src_sc + static_cast<int64_t>(ok ? t : 0) * words;
    const int c1 = min(8 * g + 8, words);
#pragma unroll 1
    for (int c = 8 * g; c < c1; c += 2) {
      const uint32_t v0 = ok ? __ldcg(row + c) : 0x7F7F7F7Fu;
      const uint32_t v1 = (ok && c + 1 < c1) ? __ldcg(row + c + 1) : 0x7F7F7F7Fu;
      dst_sc[static_cast<int64_t>(c) * n_rows + p] = v0;
      if (c + 1 < c1) dst_sc[static_cast<int64_t>(c + 1) * n_rows + p] = v1;
    }
  }
}

template <int PER>
__global__ void __launch_bounds__(kPermuteChunk) k_prologue_big(PrologueArgs a, BigPrologueArgs b) {
  extern __shared__ uint32_t bits[];
  // the GEMM after this grid waits for its completion (griddepcontrol.wait) and
  // may set up meanwhile
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned G = gridDim.x;
  const int nchunks = (a.T + kPermuteChunk - 1) / kPermuteChunk;
  // the streaming work (quantisation of x, zeroing of out) runs on the blocks
  // the permutation leaves idle (blocks >= nchunks) during its two phases,
  // or in phase 0 when there are none
  const bool spare = static_cast<int>(G) > nchunks;
  auto quantize = [&](int64_t first, int64_t stride) {
    if (a.act_e2m1)
      for (int64_t i = first; i - lane < a.n8; i += stride)
        quantize_act_step_e2m1(a.x, a.n8, i, lane, reinterpret_cast<uint32_t*>(a.codes), a.scales);
    else
      for (int64_t i = first; i - lane < a.n8; i += stride) quantize_act_step(a.x, a.n8, i, lane, a.codes, a.scales);
  };
  auto zero_out = [&](int64_t first, int64_t stride) {
    for (int64_t i = first; i < a.n_out4; i += stride) a.out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  };
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid;
  const int64_t spare_stride = static_cast<int64_t>(static_cast<int>(G) - nchunks) * blockDim.x;
  const int64_t spare_first = static_cast<int64_t>(static_cast<int>(blockIdx.x) - nchunks) * blockDim.x + tid;
  // phase 0: routing
  for (int t = blockIdx.x * (kPermuteChunk / 32) + warp; t < a.T; t += gridDim.x * (kPermuteChunk / 32))
    topk_token<PER>(a.logits, t, a.E, a.k, lane, a.ids, a.topk_w);
  if (!spare) {
    quantize(first, stride);
    zero_out(first, stride);
  }
  if (!grid_barrier(b.bar, G, a.sc.status, b.wait_limit_ns)) return;
  // phase 1: counting pass, offsets and chunk bases (last chunk block); the
  // spare blocks quantise x
  if (static_cast<int>(blockIdx.x) < nchunks)
    permute_count_block(a.ids, a.T, a.E, a.k, a.counts, a.offsets, a.sorted_slot, a.sc, nchunks, blockIdx.x, bits);
  else
    quantize(spare_first, spare_stride);
  if (!grid_barrier(b.bar, 2 * G, a.sc.status, b.wait_limit_ns)) return;
  // phase 2: scatter (as k_permute_scatter; the counters are reset for the
  // next call); the spare blocks zero out
  if (static_cast<int>(blockIdx.x) >= nchunks) zero_out(spare_first, spare_stride);
  if (static_cast<int>(blockIdx.x) < nchunks) {
    const int chunk = blockIdx.x;
    const int t = chunk * kPermuteChunk + tid;
    if (blockIdx.x == 0 && tid == 0) *a.sc.done = 0u;
    if (t < a.T) {
      for (int j = 0; j < a.k; ++j) {
        const int e = __ldcg(&a.ids[static_cast<int64_t>(t) * a.k + j]);
        if (e < 0 || e >= a.E) continue;
        const int pos = __ldcg(&a.sc.chunk_base[static_cast<int64_t>(chunk) * a.E + e]) +
                        __ldcg(&a.sc.local_rank[static_cast<int64_t>(t) * a.k + j]);
        a.sorted_slot[pos] = t * (a.k + 1) + j;
      }
      a.sorted_slot[__ldcg(&a.offsets[a.E]) + t] = t * (a.k + 1) + a.k;
    }
  }
  if (b.gathered == nullptr) return;
  if (!grid_barrier(b.bar, 3 * G, a.sc.status, b.wait_limit_ns)) return;
  // phase 3: activation rows in slot order (16-byte units; written above by
  // other blocks, so read through L2)
  // four independent copies in flight per thread (each a slot load, then a
  // row load, then a store)
  const int64_t row_chunks = b.row_bytes / 16;
  const int64_t total = row_chunks * static_cast<int64_t>(a.T) * (a.k + 1);
  const uint4* __restrict__ src = reinterpret_cast<const uint4*>(a.codes);
  uint4* __restrict__ dst = reinterpret_cast<uint4*>(b.gathered);
  const int32_t* __restrict__ ss = a.sorted_slot;
  for (int64_t i0 = first; i0 < total; i0 += 4 * stride) {
    int tt[4];
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      tt[u] = i < total ? __ldcg(&ss[i / row_chunks]) / (a.k + 1) : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < total && tt[u] >= 0 && tt[u] < a.T) v[u] = __ldcg(&src[static_cast<int64_t>(tt[u]) * row_chunks + i % row_chunks]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i >= total) continue;
      if (tt[u] < 0 || tt[u] >= a.T) set_status(a.sc.status, MX_ERR_DEVICE_ARG);
      else dst[i] = v[u];
    }
  }
  if (b.gathered_scales)
    gather_scales_t(reinterpret_cast<const uint32_t*>(a.scales), a.T, static_cast<int>(b.scale_words), ss, a.k,
                    a.T * (a.k + 1), b.gathered_scales, first, stride);
}

// Blocks of the large-batch prologue that fit on the GPU at once (0: none).
int prologue_big_blocks(const PrologueArgs& a) {
  const size_t smem = permute_block_smem(a.T, a.E, a.k);
  void (*kern)(PrologueArgs, BigPrologueArgs) = a.E <= 32 ? k_prologue_big<1> : a.E <= 128 ? k_prologue_big<4>
                                               : a.E <= 512 ? k_prologue_big<16> : k_prologue_big<32>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPermuteChunk, smem) != cudaSuccess) return 0;
  if (per_sm > 8) per_sm = 8;
  const int nchunks = (a.T + kPermuteChunk - 1) / kPermuteChunk;
  const int blocks = per_sm * sm_count();
  return blocks >= nchunks ? blocks : 0;
}

cudaError_t launch_prologue_big(const PrologueArgs& a, const BigPrologueArgs& b, int blocks, cudaStream_t s) {
  const size_t smem = permute_block_smem(a.T, a.E, a.k);
  void (*kern)(PrologueArgs, BigPrologueArgs) = a.E <= 32 ? k_prologue_big<1> : a.E <= 128 ? k_prologue_big<4>
                                               : a.E <= 512 ? k_prologue_big<16> : k_prologue_big<32>;
  // the barrier counter and the permutation's last-block counter start at
  // zero (memsets, not kernels; the latter also after an earlier call that
  // stopped half-way)
  cudaError_t e = cudaMemsetAsync(b.bar, 0, sizeof(unsigned), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.sc.done, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(blocks), kPermuteChunk, smem, s>>>(a, b);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ row gather
__global__ void __launch_bounds__(256) k_gather_rows(const uint4* __restrict__ src, int T,
                                                     int64_t row_chunks,
                                                     const int32_t* __restrict__ sorted_slot, int k,
                                                     int64_t total_chunks, uint4* __restrict__ dst,
                                                     const uint32_t* __restrict__ src_sc, int64_t scale_words,
                                                     uint32_t* __restrict__ dst_sc, int* status) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t i = first; i < total_chunks; i += stride) {
    const int64_t p = i / row_chunks, c = i - p * row_chunks;
    const int t = __ldg(&sorted_slot[p]) / (k + 1);
    if (t < 0 || t >= T) {
      set_status(status, MX_ERR_DEVICE_ARG);
      continue;
    }
    dst[i] = __ldg(&src[static_cast<int64_t>(t) * row_chunks + c]);
  }
  if (dst_sc)
    gather_scales_t(src_sc, T, static_cast<int>(scale_words), sorted_slot, k,
                    static_cast<int>(total_chunks / row_chunks), dst_sc, first, stride);
}

cudaError_t launch_gather_rows(const uint8_t* src, int T, int64_t row_bytes,
                               const int32_t* sorted_slot, int k, int n_rows, uint8_t* dst,
                               const uint32_t* src_sc, int64_t scale_words, uint32_t* dst_sc,
                               int* status, cudaStream_t s) {
  const int64_t row_chunks = row_bytes / 16;
  const int64_t total = row_chunks * n_rows;
  if (total == 0) return cudaSuccess;
  k_gather_rows<<<grid_for(total, 256, 8), 256, 0, s>>>(reinterpret_cast<const uint4*>(src), T,
                                                        row_chunks, sorted_slot, k, total,
                                                        reinterpret_cast<uint4*>(dst), src_sc, scale_words,
                                                        dst_sc, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ weight re-layout
// Block (e, kc, rb') of 128 rows x 128 K elements sits at linear index
// (e * NK + kc) * RB + rb': for one K chunk, all row blocks of an expert are
// adjacent, so the two row blocks a GEMM tile multiplies (gate block m and up
// block m, interleaved as rb' = 2m and 2m + 1 in W1; row blocks 2m and 2m + 1 in
// W2) arrive with one TMA box.
PreparedLayout prepared_layout(int E1, int rows, int K, int fmt, int interleave) {
  PreparedLayout L;
  L.E1 = E1;
  L.rows = rows;
  L.K = K;
  L.fmt = fmt;
  L.RB = rows / 128;
  L.NK = K / 128;
  L.interleave = interleave;
  L.block_code_bytes = fmt == MX_E4M3 ? 16384 : 8192;
  const size_t nblk = static_cast<size_t>(E1) * L.RB * L.NK;
  L.codes_bytes = nblk * L.block_code_bytes;
  L.scales_offset = (L.codes_bytes + 1023) & ~static_cast<size_t>(1023);
  L.scales_bytes = nblk * 512;
  L.total_bytes = L.scales_offset + L.scales_bytes;
  return L;
}

// canonical row block of prepared row block rb'
__device__ __forceinline__ int canonical_rb(int rbp, int RB, int interleave) {
  return interleave ? ((rbp & 1) ? RB / 2 + (rbp >> 1) : (rbp >> 1)) : rbp;
}

// codes: one thread per 16-byte chunk of the destination block
__global__ void __launch_bounds__(256) k_prepare_codes(const uint4* __restrict__ src, int rows,
                                                       int64_t src_row_chunks, int RB, int NK, int interleave,
                                                       int blk_row_chunks, int64_t total,
                                                       uint4* __restrict__ dst) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t per_blk = static_cast<int64_t>(128) * blk_row_chunks;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t b = i / per_blk;
    const int within = static_cast<int>(i - b * per_blk);
    const int r = within / blk_row_chunks, c = within - r * blk_row_chunks;
    const int rbp = static_cast<int>(b % RB);
    const int64_t ekc = b / RB;
    const int kc = static_cast<int>(ekc % NK);
    const int64_t e = ekc / NK;
    const int rb = canonical_rb(rbp, RB, interleave);
    const int64_t src_row = e * rows + static_cast<int64_t>(rb) * 128 + r;
    dst[i] = __ldg(&src[src_row * src_row_chunks + static_cast<int64_t>(kc) * blk_row_chunks + c]);
  }
}

// scales: one thread per 32-bit word of a 512-byte block: lane l, word j holds
// the four k-blocks of row 32*j + l (the tensor-memory scale-factor layout of
// the block-scaled MMA: a lane's 16-byte word is what it stores into its
// tensor-memory lane with tcgen05.st 32x32b.x4).
__global__ void __launch_bounds__(256) k_prepare_scales(const uint8_t* __restrict__ src, int rows,
                                                        int K32, int RB, int NK, int interleave,
                                                        int64_t total_words, uint32_t* __restrict__ dst) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_words;
       i += stride) {
    const int64_t b = i / 128;
    const int w = static_cast<int>(i & 127);
    const int l = w >> 2, j = w & 3;
    const int rbp = static_cast<int>(b % RB);
    const int64_t ekc = b / RB;
    const int kc = static_cast<int>(ekc % NK);
    const int64_t e = ekc / NK;
    const int rb = canonical_rb(rbp, RB, interleave);
    const int64_t row = e * rows + static_cast<int64_t>(rb) * 128 + 32 * j + l;
    dst[i] = __ldg(reinterpret_cast<const uint32_t*>(src + row * K32 + static_cast<int64_t>(kc) * 4));
  }
}

cudaError_t launch_prepare_weights(const uint8_t* codes, const uint8_t* scales,
                                   const PreparedLayout& L, uint8_t* dst, cudaStream_t s) {
  const int64_t nblk = static_cast<int64_t>(L.E1) * L.RB * L.NK;
  const int blk_row_chunks = L.fmt == MX_E4M3 ? 8 : 4;
  const int64_t src_row_chunks = (L.fmt == MX_E4M3 ? L.K : L.K / 2) / 16;
  const int64_t total = nblk * 128 * blk_row_chunks;
  if (total > 0) {
    k_prepare_codes<<<grid_for(total, 256, 8), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(codes), L.rows, src_row_chunks, L.RB, L.NK, L.interleave,
        blk_row_chunks, total, reinterpret_cast<uint4*>(dst));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t words = nblk * 128;
    k_prepare_scales<<<grid_for(words, 256, 8), 256, 0, s>>>(
        scales, L.rows, L.K / 32, L.RB, L.NK, L.interleave, words,
        reinterpret_cast<uint32_t*>(dst + L.scales_offset));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s) {
  return cudaMemsetAsync(p, 0, bytes, s);
}

}  // namespace mxk
