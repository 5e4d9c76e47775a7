// Device helpers shared by the MX MoE kernels: MX block-exponent extraction
// and round-to-nearest-even encoders for E4M3 / E2M1, written from the element
// definitions of the OCP Microscaling Formats (MX) v1.0 specification.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/mxmoe.h"

namespace mxk {

// floor(log2(a)) for a finite a > 0 given its fp32 bit pattern (sign cleared);
// fp32 subnormals are m * 2^-149.
__device__ __forceinline__ int floor_log2_bits(uint32_t a) {
  const int ef = static_cast<int>(a >> 23);
  if (ef > 0) return ef - 127;
  return -149 + (31 - __clz(a & 0x7FFFFFu));
}

// Shared block exponent s = clamp(floor(log2(amax)) - emax, -127, 127); an
// all-zero block (amax = 0, log2 = -inf) takes the lower clamp.
__device__ __forceinline__ int mx_block_exponent(uint32_t amax_bits, int emax) {
  if (amax_bits == 0u) return -127;
  int s = floor_log2_bits(amax_bits) - emax;
  return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// 2^-s as an fp32 for s in [-127, 126] (exact power of two).
__device__ __forceinline__ float pow2_neg(int s) {
  return __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
}

// E4M3 code of q (finite, |q| < 512 after block scaling): round to nearest
// even on the E4M3 grid (subnormal spacing 2^-9 below 2^-6), saturate at 448
// (0x7E), keep the sign of q (so a negative value rounding to zero is 0x80).
__device__ __forceinline__ uint32_t enc_e4m3(float q) {
  const uint32_t u = __float_as_uint(q);
  const uint32_t sign = (u >> 24) & 0x80u;
  const uint32_t a = u & 0x7FFFFFFFu;
  uint32_t code;
  if (a >= 0x43E00000u) {            // >= 448
    code = 0x7Eu;
  } else if (a < 0x3C800000u) {      // < 2^-6: code = round(a / 2^-9), 0..8
    code = static_cast<uint32_t>(__float2int_rn(__uint_as_float(a) * 512.0f));
  } else {                           // normal: keep 3 mantissa bits, ties to even
    const uint32_t r = (a + 0x7FFFFu + ((a >> 20) & 1u)) >> 20;
    code = r - 960u;                 // (biased fp32 exponent - 120) << 3 | mantissa
  }
  return sign | code;
}

// E2M1 code of q (finite, |q| < 8): magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6;
// the thresholds are the midpoints, a midpoint going to the even code.
__device__ __forceinline__ uint32_t enc_e2m1(float q) {
  const float a = fabsf(q);
  const uint32_t code = static_cast<uint32_t>(a > 0.25f) + static_cast<uint32_t>(a >= 0.75f) +
                        static_cast<uint32_t>(a > 1.25f) + static_cast<uint32_t>(a >= 1.75f) +
                        static_cast<uint32_t>(a > 2.5f) + static_cast<uint32_t>(a >= 3.5f) +
                        static_cast<uint32_t>(a > 5.0f);
  return ((__float_as_uint(q) >> 28) & 8u) | code;
}

__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

}  // namespace mxk
