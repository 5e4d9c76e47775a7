// Device helpers shared by the MX MoE kernels: MX block-exponent extraction
// and round-to-nearest-even encoders for E4M3 / E2M1, written from the element
// definitions of the OCP Microscaling Formats (MX) v1.0 specification.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/mxmoe.h"

namespace mxk {

// Shared block exponent s = clamp(floor(log2(amax)) - emax, -127, 127) for a
// finite amax given as fp32 bits with the sign cleared, emax >= 0.  Written
// without branches: a normal amax has floor(log2) = biased exponent - 127; a
// subnormal or zero amax (biased exponent 0, log2 below -126, or -inf for 0)
// always lands at the lower clamp, and so does the formula with exponent 0;
// the upper clamp is never reached (biased exponent <= 254, emax >= 0).
__device__ __forceinline__ int mx_block_exponent(uint32_t amax_bits, int emax) {
  return max(static_cast<int>(amax_bits >> 23) - 127 - emax, -127);
}

// 2^-s as an fp32 for s in [-127, 126] (exact power of two).
__device__ __forceinline__ float pow2_neg(int s) {
  return __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
}

// E4M3 codes of two block-scaled values (finite) with the hardware conversion:
// round to nearest even on the E4M3 grid (subnormal spacing 2^-9 below 2^-6),
// saturate at 448 (0x7E), keep the sign (a negative value rounding to zero is
// 0x80).  The code of `lo` is in bits 0..7, that of `hi` in bits 8..15.
__device__ __forceinline__ uint32_t enc_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
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
