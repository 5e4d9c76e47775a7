// moe_permute_no_alloc: the token -> expert permutation for callers that
// cannot hand the library any device memory of its own to use as scratch.
//
// Who needs this: code that runs where allocating is not allowed or not
// possible -- a plugin whose host framework owns every device allocation and
// forbids cudaMalloc inside its enqueue callback, or a serving loop that must
// not allocate on the hot path because cudaMalloc/cudaFree can synchronise the
// device.  Such callers still own the inputs and outputs; only the scratch moves
// into the library.
//
// The scratch is one file-scope device array of fixed size that every call on a
// device shares.  Consequences for callers:
//   * requests whose scratch would exceed kNoAllocScratchBytes are rejected
//     with MX_ERR_WORKSPACE before anything is enqueued;
//   * two calls that overlap on the GPU (different streams, no ordering between
//     them) race on the shared array -- order them on one stream;
//   * the first call on each device looks the array's device address up
//     (cudaGetSymbolAddress with that device current) and caches it; make that
//     first call before any stream capture begins.
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "../../include/mxmoe.h"
#include "internal.h"

namespace {

// Enough for T <= 8192 tokens, E <= 512 experts, k <= 8 (393,728 bytes needed).
constexpr size_t kNoAllocScratchBytes = 400 * 1024;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device.  In host code the
// array's name is only a handle for the runtime: the address the kernels need
// comes from cudaGetSymbolAddress, looked up once per device.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MX_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MX_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return MX_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MX_OK;
}

}  // namespace

extern "C" MX_API int moe_permute_no_alloc(const int32_t* topk_ids, int T, int E, int k,
                                           int32_t* counts, int32_t* offsets,
                                           int32_t* sorted_slot, mx_stream_t stream) {
  if (T < 0 || E <= 0 || k < 1 || k > E || k > 32) return MX_ERR_INVALID_ARG;
  if (E > 1024) return MX_ERR_UNSUPPORTED;
  if (!counts || !offsets || (T > 0 && (!topk_ids || !sorted_slot))) return MX_ERR_INVALID_ARG;
  const size_t need = mxk::permute_scratch_bytes(T, E, k);
  if (need > kNoAllocScratchBytes) return MX_ERR_WORKSPACE;
  void* base = nullptr;
  const int st = scratch_address(&base);
  if (st != MX_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const mxk::PermuteScratch sc = mxk::permute_scratch_carve(base, T, E, k);
  // the array keeps the previous call's contents: the status word and the
  // last-block counter must start at zero
  if (cudaMemsetAsync(sc.status, 0, sizeof(int), s) != cudaSuccess) return MX_ERR_CUDA;
  if (cudaMemsetAsync(sc.done, 0, sizeof(unsigned), s) != cudaSuccess) return MX_ERR_CUDA;
  return mxk::launch_permute(topk_ids, T, E, k, counts, offsets, sorted_slot, sc, s) == cudaSuccess
             ? MX_OK
             : MX_ERR_CUDA;
}
