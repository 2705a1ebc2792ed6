// fp8block.cuh -- the blockwise FP8 scale rule (device helper shared by the quantise
// kernels and the row permutation that quantises as it copies).
//
// A block's scale is 2^ceil(log2(amax / 448)): the smallest power of two that keeps
// every element within E4M3's +-448 (2^-127 for an all-zero block, exponents clipped
// to [-127, 127]).
#pragma once
#include <cstdint>

namespace mmmoe {
namespace fb {

constexpr int FB = 128;  // block length

// ceil(log2(amax / 448)) clipped to [-127, 127], -127 for amax = 0.  With amax =
// m * 2^E (m in [1, 2)) and 448 = 1.75 * 2^8 it is E - 8, plus 1 when m > 1.75.
__device__ __forceinline__ int ceil_exp(float amax) {
  if (!(amax > 0.f)) return -127;
  const uint32_t b = __float_as_uint(amax);
  const int e = static_cast<int>((b >> 23) & 0xFFu) - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u);
  return max(-127, min(127, e));
}

}  // namespace fb
}  // namespace mmmoe
