// Order-preserving 32-bit keys of fp32 values for warp-wide top-k selection:
// the key of a larger value is a larger unsigned integer, so a round's winner
// is one warp reduction (redux.sync max) away, and the lowest index holding it
// a second (min).  -0 is folded into +0 first, so values that compare equal as
// floats get equal keys; key 0 lies below every value's key (-inf's included)
// and marks an empty slot.
#pragma once
#include <cstdint>

namespace mxk {

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t b = __float_as_uint(x + 0.0f);  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

}  // namespace mxk
