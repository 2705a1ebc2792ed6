// mx.cuh -- MXFP8 block quantisation of single values (device helpers shared by the
// quantise kernels and the GEMM epilogues that emit quantised operands).
//
// OCP Microscaling v1.0 MXFP8: a block of 32 elements shares the power-of-two scale
// 2^(floor(log2 amax) - 8) (8 = the largest E4M3 exponent; 2^-127 for an all-zero
// block); an element is v / scale rounded to E4M3 (nearest even, saturating at
// +-448).  The helpers return the dequantised value e4m3 * scale, which bf16 holds
// exactly.  The quantised input is always the bf16 value the layer stores.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace mmmoe {
namespace mx {

// Shared-scale exponent of a block with absolute maximum amax (>= 0).
__device__ __forceinline__ int scale_exp(float amax) {
  if (!(amax > 0.f)) return -127;
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 8;
  return max(-127, min(127, e));  // a subnormal amax gives a very negative e: clamp
}

// 2^k for k in [-127, 127], exactly (2^-127 is an fp32 subnormal; the library is
// built without flush-to-zero).
__device__ __forceinline__ float pow2f(int k) {
  return k >= -126 ? __uint_as_float(static_cast<uint32_t>(k + 127) << 23)
                   : __uint_as_float(0x00400000u);
}

// Dequantised E4M3 values of a pair under block exponents ea, eb.  Scaling by a
// power of two is exact here (|v| / 2^e < 512, and e4m3 * 2^e >= 2^-136 is an fp32
// value), so the only rounding is the E4M3 conversion.
__device__ __forceinline__ void qdq2(float& a, float& b, int ea, int eb) {
  const __nv_fp8x2_storage_t s = __nv_cvt_float2_to_fp8x2(
      make_float2(a * pow2f(-ea), b * pow2f(-eb)), __NV_SATFINITE, __NV_E4M3);
  const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(s, __NV_E4M3)));
  a = f.x * pow2f(ea);
  b = f.y * pow2f(eb);
}

// bf16 bit pattern <-> value
__device__ __forceinline__ float bf(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t to_bf(float f) {
  const __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<const uint16_t*>(&h);
}
// v rounded to bf16, as a float
__device__ __forceinline__ float round_bf(float f) { return bf(to_bf(f)); }

// ---------------------------------------------------------------- MXFP8 storage
// The block-scaled tensor cores read an MXFP8 operand as e4m3 codes (one byte per
// element, in the operand's own row-major layout) and E8M0 scale codes (2^e stored as
// e + 127; all-zero blocks store 0, i.e. 2^-127) in the arrangement below.  For an
// operand whose MMA rows (rows of A, or of B) are indexed by mn and whose K is cut
// into 32-element k-blocks kb: 512-byte atoms of 128 consecutive mn x 4 consecutive
// kb; inside an atom, mn % 32 picks a 16-byte row, (mn / 32) % 4 a 4-byte word of it
// and kb % 4 the byte of the word; the atoms of one group of 4 k-blocks lie side by
// side for consecutive 128-row blocks of mn (mn_blocks of them), then the next group.
// A GEMM stage (128 elements of K) then reads one atom per 128 rows of each operand.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t mn, int64_t kb, int64_t mn_blocks) {
  return ((kb >> 2) * mn_blocks + (mn >> 7)) * 512 + (mn & 31) * 16 + ((mn >> 5) & 3) * 4 +
         (kb & 3);
}

// E8M0 code of the block scale 2^e (e in [-127, 127]).
__device__ __forceinline__ uint32_t e8m0(int e) { return static_cast<uint32_t>(e + 127); }

// e4m3 codes of v / 2^e for two values (nearest even, saturating at +-448); a in the
// low byte.  Exact scaling as in qdq2.
__device__ __forceinline__ uint32_t codes2(float a, float b, int e) {
  const float s = pow2f(-e);
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(a * s, b * s), __NV_SATFINITE, __NV_E4M3));
}

// Eight values under one exponent -> eight codes (element 0 in the lowest byte).
__device__ __forceinline__ uint2 codes8(const float (&v)[8], int e) {
  return make_uint2(codes2(v[0], v[1], e) | (codes2(v[2], v[3], e) << 16),
                    codes2(v[4], v[5], e) | (codes2(v[6], v[7], e) << 16));
}

// One thread's 32 values form one block: round them to bf16 (the stored value),
// return the block exponent and the 32 codes (4 x 8 bytes).
__device__ __forceinline__ int quant_row32(const float (&v)[32], uint2 (&out)[4]) {
  float r[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    r[i] = round_bf(v[i]);
    amax = fmaxf(amax, fabsf(r[i]));
  }
  const int e = scale_exp(amax);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = r[8 * q + j];
    out[q] = codes8(w, e);
  }
  return e;
}

// Scale exponent of a block whose largest absolute value has the bf16 bit pattern
// `bits` (sign clear): floor(log2) - 8 from the exponent field, -127 for zero, and
// clamped to [-127, 127] like scale_exp (a subnormal maximum gives -127).
__device__ __forceinline__ int bf16_scale_exp(uint32_t bits) {
  const int ef = static_cast<int>((bits >> 7) & 0xFFu);
  return ef == 0 ? -127 : max(-127, ef - 127 - 8);
}

// Four e4m3 codes of the bf16 values in two words (element 0 in the low half of w0),
// each times its own power-of-two multiplier (exact); element 0's code in the lowest
// byte.
__device__ __forceinline__ uint32_t codes4(uint32_t w0, uint32_t w1, float m0, float m1,
                                           float m2, float m3) {
  const float a = __uint_as_float(w0 << 16), b = __uint_as_float(w0 & 0xFFFF0000u);
  const float c = __uint_as_float(w1 << 16), d = __uint_as_float(w1 & 0xFFFF0000u);
  const uint32_t lo = static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(a * m0, b * m1), __NV_SATFINITE, __NV_E4M3));
  const uint32_t hi = static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(c * m2, d * m3), __NV_SATFINITE, __NV_E4M3));
  return lo | (hi << 16);
}

}  // namespace mx
}  // namespace mmmoe
