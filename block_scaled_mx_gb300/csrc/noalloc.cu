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
//     first call before any stream capture begins.  The cache is keyed on the
//     device's current CUDA context, so after cudaDeviceReset (a new context,
//     a new address) the next call looks the address up again.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
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
struct CachedAddress {
  unsigned long long ctx_id;  // context the address belongs to (0: none cached)
  void* addr;
};
CachedAddress g_scratch_addr[kMaxDevices] = {};

// Process-unique id of the calling thread's current CUDA context, or 0 when it
// cannot be had (then nothing is cached).  The driver calls come through the
// runtime's entry-point query, so the library needs no link against libcuda.
unsigned long long current_context_id(int dev) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) {
    // no context current on this thread yet: make the device's primary
    // context current (what the runtime would do on its first call)
    if (cudaSetDevice(dev) != cudaSuccess || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  }
  unsigned long long id = 0;
  return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_permute_scratch on the current device.  In host code the
// array's name is only a handle for the runtime: the address the kernels need
// comes from cudaGetSymbolAddress, looked up once per device and context.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MX_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MX_ERR_UNSUPPORTED;
  const unsigned long long ctx = current_context_id(dev);
  std::lock_guard<std::mutex> lock(g_mu);
  CachedAddress& c = g_scratch_addr[dev];
  if (ctx == 0 || c.ctx_id != ctx || !c.addr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return MX_ERR_CUDA;
    c.addr = p;
    c.ctx_id = ctx;
  }
  *out = c.addr;
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
